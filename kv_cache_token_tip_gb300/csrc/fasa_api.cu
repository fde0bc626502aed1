// Host side of the C ABI: argument validation, shared-memory planning,
// cluster sizing and launches; plus the small auxiliary kernels (query RoPE,
// dominant-key copy build and append).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/fasa.h"
#include "fasa_cluster.cuh"
#include "fasa_internal.h"

using namespace fasa;

namespace {

__device__ int g_status;  // FASA_DEV_* bits, per device

thread_local int t_last_cuda_error = 0;

// Bound of every device wait (fasa_test_fault_injection can shorten it) and
// the test hook that leaves one TIP tile's copy unissued (-1: none).
unsigned long long g_wait_ns = 1000000000ull;
int g_drop_tip_tile = -1;
int g_drop_fac_refill = -1;


int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return FASA_ERR_CUDA;
}

constexpr int SMEM_LIMIT = 232448;  // 227 KB per CTA
constexpr int S_CAP_MAX = 8192;     // scores per CTA kept in shared memory
constexpr int STEP_MIN_C = 4;       // smallest cluster the single-exchange step kernel serves

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int align_up(int x, int a) { return (x + a - 1) / a * a; }
int ceil_div(int a, int b) { return (a + b - 1) / b; }

int check_dims(const fasa_dims_t* d) {
  if (!d) return FASA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1) return FASA_ERR_INVALID_ARG;
  if (d->n_q_heads % d->n_kv_heads) return FASA_ERR_INVALID_ARG;
  if (d->head_dim < 2 || (d->head_dim & 1)) return FASA_ERR_INVALID_ARG;
  if (d->t_max < 1 || (d->t_max % KDOM_BLOCK)) return FASA_ERR_INVALID_ARG;
  if (d->n_tip < 1 || d->n_tip > d->head_dim / 2) return FASA_ERR_INVALID_ARG;
  if (!(d->rope_theta > 0.0) || !isfinite(d->rope_theta)) return FASA_ERR_INVALID_ARG;
  if (d->reserved < 0 || d->reserved > C_MAX) return FASA_ERR_INVALID_ARG;
  if (d->dtype != FASA_F32 && d->dtype != FASA_BF16) return FASA_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return FASA_ERR_UNSUPPORTED;
  if (d->n_q_heads / d->n_kv_heads > G_MAX) return FASA_ERR_UNSUPPORTED;
  if ((long long)d->batch * d->n_kv_heads > 65535) return FASA_ERR_UNSUPPORTED;
  return FASA_OK;
}

int elem_size(const fasa_dims_t* d) { return d->dtype == FASA_F32 ? 4 : 2; }

struct DevInfo {
  int sms = 0;
  int smem_optin = 0;
  int* status = nullptr;
};

int device_info(DevInfo* out) {
  static std::mutex mu;
  static std::map<int, DevInfo> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    DevInfo di;
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (di.smem_optin > SMEM_LIMIT) di.smem_optin = SMEM_LIMIT;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.status), g_status);
    if (e != cudaSuccess) return cuda_fail(e);
    it = cache.emplace(dev, di).first;
  }
  *out = it->second;
  return FASA_OK;
}

// How many clusters of C CTAs with `smem` bytes each can be resident at once
// (0: the cluster cannot be launched).  Cached per configuration.
int cluster_capacity(int flags, int dtype, int D, int C, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const int kind = kind_of(flags);
  const auto key = std::make_tuple(dev, kind, dtype, D, C, smem);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const int n = dtype == FASA_F32 ? max_active_clusters_f32(flags, D, C, smem)
                                  : max_active_clusters_bf16(flags, D, C, smem);
  cache.emplace(key, n);
  return n;
}

// Shared-memory plan of one launch (byte offsets into dynamic shared memory).
//
// Persistent regions: mbarriers, scratch, rotated queries, the query restricted
// to the dominant FCs, the tile logits, the local and cluster histograms, the
// CTA's scores, the selected-index list, this CTA's candidate list (read by
// the other CTAs) and the partial attention record (read by the combining
// CTA).  The "big" region is the TIP ring during the scan, then the pulled
// candidate list followed by the FAC ring.
//
// Returns FASA_OK, or FASA_ERR_UNSUPPORTED when it cannot fit in `limit`
// bytes.  *ws = global workspace bytes needed.
int plan_smem(Params& p, const fasa_dims_t* d, int C, int flags, bool allow_ws, size_t* ws, int limit) {
  const int D = d->head_dim, es = elem_size(d), G = d->n_q_heads / d->n_kv_heads;
  const int nfc = d->n_tip;
  const bool select = (flags & F_SELECT) != 0;
  const bool tip = (flags & F_TIP) != 0;
  const bool fac = (flags & (F_FAC | F_DENSE)) != 0;
  int off = 0;
  p.off_bar = off;
  off += 64;  // mbarriers of the TIP ring
  p.off_misc = off;
  off += MISC_BYTES;
  p.off_qrot = off;
  off += G_MAX * D * 4;
  p.off_qbar = off;
  off += align_up(2 * nfc * 4, 16);
  p.off_stile = off;
  off += (es == 2 ? NW * G_MAX * PTS : G_MAX * RT) * 4;
  p.off_hloc = off;
  off += select ? HLOC_BINS * 4 : 0;
  p.off_hlead = off;
  off += select ? HLEAD_BINS * 4 : 0;
  // given indices (F_IDX_IN) are staged per CTA; selections live in the candidate list
  p.idx_cap = (flags & F_IDX_IN) ? align_up(p.budget, 4) : 0;
  p.hpc = ceil_div(G, C);
  const int part_bytes = fac ? G * (D + 4) * 4 : 0;
  // pushed partial records: [C][largest slice] float4 groups, then [C][G] (m, l)
  const int ngrp4 = G * (D / 4);
  const int recv_bytes = fac ? align_up(C * ceil_div(ngrp4, C) * 16 + C * G * 8, 128) : 0;
  // FAC staging: fp32 -- a block-wide ring of FAC_STAGES tiles of RT padded
  // rows; bf16 -- per warp, wst slots of one GR-row group of swizzled rows
  // (two slots if they fit)
  auto fac_bytes = [&](int wst) {
    if (!fac) return 0;
    return es == 2 ? wst * NW * 2 * GR * (D * es) : FAC_STAGES * 2 * RT * (D * es + 16);
  };

  int s_cap = 0;
  *ws = 0;
  if (tip && select) {
    const int chunk = align_up(ceil_div(d->t_max, C), KDOM_BLOCK);
    if (chunk <= S_CAP_MAX) s_cap = chunk;
  }
  // preference: scores in shared memory before two groups in flight per warp
  const int s_cap0 = s_cap;
  for (int attempt = 0; attempt < 4; ++attempt) {
    const int wst = (es == 2 && attempt % 2 == 0) ? 2 : 1;
    if (attempt % 2 == 1 && es != 2) continue;  // fp32 has no per-warp groups
    if (attempt >= 2 && s_cap0 == 0) break;     // no second layout of the scores
    s_cap = attempt < 2 ? s_cap0 : 0;
    const int fac_big = fac_bytes(wst);
    p.fac_wst = wst;
    int o = off;
    p.off_sc = o;
    o += s_cap * 4;
    p.off_idx = o;
    o += p.idx_cap * 4;
    // candidate capacity: the budget plus as much slack (up to 4096) as fits
    // next to the FAC ring
    int cap = 0;
    if (select) {
      cap = (limit - (o + part_bytes + recv_bytes + 384) - fac_big) / 8;
      if (cap > p.budget + 4096) cap = p.budget + 4096;
      cap &= ~15;
    }
    p.cand_cap = cap;
    p.off_own = o;
    o += cap * 8;
    p.off_part = o;
    o += part_bytes;
    o = align_up(o, 128);
    p.off_recv = o;
    o += recv_bytes;
    o = align_up(o, 128);
    p.off_big = o;
    p.fac_off = 0;
    int bigsz = fac_big;
    int tile = 256, stages = 1;
    if (tip) {
      // the largest tile with at least two stages in the room left, up to a
      // ring of 4 stages / 128 KB
      const int tiles[3] = {1024, 512, 256};
      for (int ti = 0; ti < 3; ++ti) {
        const int stage = nfc * tiles[ti] * 2 * es;
        int st = 131072 / stage;
        st = st < 1 ? 1 : (st > 4 ? 4 : st);
        while (st > 1 && o + (st * stage > bigsz ? st * stage : bigsz) > limit) --st;
        tile = tiles[ti];
        stages = st;
        if (st >= 2) break;
      }
      const int stage = nfc * tile * 2 * es;
      if (stages * stage > bigsz) bigsz = stages * stage;
    }
    p.tip_tile = tile;
    p.tip_stages = stages;
    p.smem_total = o + bigsz;
    const bool ok = p.smem_total <= limit && (!select || cap >= p.budget);
    if (ok) {
      p.s_cap = s_cap;
      if (tip && select && s_cap == 0) {
        if (!allow_ws) return FASA_ERR_UNSUPPORTED;
        *ws = (size_t)d->batch * d->n_kv_heads * d->t_max * 4;
      }
      return FASA_OK;
    }
  }
  return FASA_ERR_UNSUPPORTED;
}

// theta_i / (2 pi) as 64-bit fixed-point turns, theta_i = B^(-2i/d)
// (cached for the last base and head dim).
void fill_rope_turns(Params& p, const fasa_dims_t* d) {
  static std::mutex mu;
  static double c_theta = -1.0;
  static int c_dim = -1;
  static unsigned long long c_turns[64];
  std::lock_guard<std::mutex> lk(mu);
  if (c_theta != d->rope_theta || c_dim != d->head_dim) {
    const long double two64_over_2pi = 18446744073709551616.0L / (2.0L * 3.14159265358979323846264338327950288L);
    for (int i = 0; i < d->head_dim / 2 && i < 64; ++i) {
      const double th = pow(d->rope_theta, -2.0 * i / d->head_dim);
      c_turns[i] = (unsigned long long)((long double)th * two64_over_2pi);
    }
    c_theta = d->rope_theta;
    c_dim = d->head_dim;
  }
  memcpy(p.rope_turns, c_turns, sizeof(c_turns));
}

void fill_common(Params& p, const fasa_dims_t* d, int32_t budget, int* status) {
  memset(&p, 0, sizeof(p));
  p.B = d->batch;
  p.Hq = d->n_q_heads;
  p.Hkv = d->n_kv_heads;
  p.G = d->n_q_heads / d->n_kv_heads;
  p.T_max = d->t_max;
  p.n_tip = d->n_tip;
  p.budget = budget;
  fill_rope_turns(p, d);
  p.status = status;
  p.wait_ns = g_wait_ns;
  p.drop_stage = g_drop_tip_tile;
}

// Plans and launches the cluster kernel.  Cluster size: the explicit
// override (dims->reserved), else the largest C (at most 16) for which every
// unit's cluster is resident at once (one wave); when no C gives one wave,
// the smallest C that can be launched for a step with a top-k, else the
// largest C <= 4.
int plan_and_launch(Params& p, const fasa_dims_t* d, int flags, void* ws, size_t ws_bytes, bool launch,
                    size_t* ws_need, int* C_out, cudaStream_t stream) {
  DevInfo di;
  int st = device_info(&di);
  if (st) return st;
  p.status = di.status;
  p.flags = flags;
  const int units = d->batch * d->n_kv_heads;
  int C = 0;
  size_t need = 0;
  if (d->reserved > 0) {
    st = plan_smem(p, d, d->reserved, flags, true, &need, di.smem_optin);
    if (st) return st;
    if (cluster_capacity(flags, d->dtype, d->head_dim, d->reserved, p.smem_total) < 1) return FASA_ERR_UNSUPPORTED;
    C = d->reserved;
  } else {
    for (int c = C_MAX; c >= 1 && !C; --c) {
      if (plan_smem(p, d, c, flags, true, &need, di.smem_optin) != FASA_OK) continue;
      if (cluster_capacity(flags, d->dtype, d->head_dim, c, p.smem_total) >= units) C = c;
    }
    // Several waves either way.  With a top-k: the fewest CTAs per unit (a
    // larger cluster only repeats the per-CTA fixed costs of the selection).
    // Without (dense or given indices: pure streaming): the largest C <= 4,
    // whose finer work units balance the waves.
    const bool sel = (flags & F_SELECT) != 0;
    for (int i = 0; i < 4 && !C; ++i) {
      const int c = sel ? 1 + i : 4 - i;
      if (plan_smem(p, d, c, flags, true, &need, di.smem_optin) != FASA_OK) continue;
      if (cluster_capacity(flags, d->dtype, d->head_dim, c, p.smem_total) >= 1) C = c;
    }
    if (!C) return FASA_ERR_UNSUPPORTED;
    st = plan_smem(p, d, C, flags, true, &need, di.smem_optin);
    if (st) return st;
  }
  if (ws_need) *ws_need = need;
  if (C_out) *C_out = C;
  if (!launch) return FASA_OK;
  if (need > 0) {
    if (!ws || ws_bytes < need || !aligned16(ws)) return FASA_ERR_WORKSPACE;
    p.scores = reinterpret_cast<float*>(ws);
  }
  const cudaError_t e = d->dtype == FASA_F32 ? launch_cluster_f32(p, d->head_dim, C, stream)
                                             : launch_cluster_bf16(p, d->head_dim, C, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FASA_OK;
}

// ------------------------------------------------------- bf16 fused step
// Shared-memory plan of the step kernel (fasa_step.cuh) for cluster size C.
//
// Persistent regions: mbarriers, scratch, rotated queries, q-bar, the digit
// histograms, the CTA's scores (when its range fits), the first-round
// receive slots (C x cap1 packed entries), the own selection, and the
// combine's receive slices.  The "big" region is the TIP staging (every
// tile of the range at once when it fits, else a ring), then the FAC
// staging, the second-round receive slots and the warp records.
//
// Returns FASA_OK, or FASA_ERR_UNSUPPORTED when it does not fit in `limit`.
// floor(2^32 / d) (0xffffffff for d = 1): q = mulhi(n, m) is n / d or one
// less for every n < 2^31, which one comparison corrects.
uint32_t div_magic(uint32_t d) { return d <= 1 ? 0xffffffffu : (uint32_t)((1ull << 32) / d); }

int plan_step(StepParams& p, const fasa_dims_t* d, int C, size_t* ws, int limit) {
  const int D = d->head_dim, G = d->n_q_heads / d->n_kv_heads, nfc = d->n_tip, k = p.budget;
  constexpr int ES = 2;
  const int chunkT = align_up(ceil_div(d->t_max, C), KDOM_BLOCK);
  // first-round list: k/C plus four standard deviations of a random share
  // (a single CTA lists its exact top k); receive slack for the rest of the
  // threshold's digit-0 bucket
  const double e = (double)k / C;
  int rho = C == 1 ? k : (int)ceil(e + 4.0 * sqrt(e) + 4.0);
  rho = std::max(1, std::min(rho, chunkT));
  // (slack for the whole threshold bin, which grows with the scores per CTA:
  // with tens of thousands a 12-bit bin near the list's end holds hundreds
  // of keys, and a list that cannot take it is refined with two more
  // histogram sweeps)
  const int cap1 = align_up(rho + std::max(std::max(64, rho / 4), chunkT / 128), 16);
  const int cap2 = C == 1 ? 0 : align_up(k + std::max(32, k / 8), 16);
  const int s_cap = chunkT <= S_CAP_MAX ? chunkT : 0;
  const int rows_cap = std::min(k, std::max(cap1, cap2));
  const int ngrp4 = G * (D / 4);
  const int sl = ceil_div(ngrp4, C);
  int off = 0;
  p.off_bar = off;
  off += ST_BARS * 8;
  p.off_fbar = off;  // the FAC slots' full and empty barriers
  off += 2 * FNW * FAC_WST_MAX * 8;
  p.off_misc = off;
  off += ST_MISC_BYTES;
  p.off_qrot = off;  // the rotated query, then the FAC's query fragments over it
  off += std::max(G * D * 4, (D / 16) * 32 * 16);
  p.off_qbar = off;
  off += align_up(2 * nfc * 4, 16);
  p.off_uh = off;
  off += UH_BINS * 4;
  p.off_rows = off;
  off += align_up(rows_cap * 4, 16);
  const int comb_slot = sl * 16 + align_up(G * 8, 16);
  p.off_comb = off;
  off += C * comb_slot;
  p.off_comb_snd = off;
  off += C * comb_slot;
  // the selection's regions, dead once the own selection is compacted, sit
  // right before `big`: a gather after the selection may use them too
  off = align_up(off, 128);
  p.off_hist = off;
  off += HLOC_BINS * 4;
  p.off_sc = off;
  off += s_cap * 4;
  p.off_recv1 = off;
  off += C * (cap1 + 2) * 8;  // per source: a 16-byte header, then the entries
  off = align_up(off, 128);
  p.off_big = off;
  const int room = limit - off;
  if (room <= 0) return FASA_ERR_UNSUPPORTED;
  // after TIP: FAC slots (then the P tiles), the second-round slots (written
  // only once every CTA drained its gathers), the warp records
  auto fac_slots = [&](int wst) { return wst * FNW * 2 * GR * D * ES; };
  const int pt_bytes = FNW * G * PTS * 4;  // each attending warp's P tile, heads x PTS
  const int rec_bytes = (G_MAX * FNW * (D + 2) + G_MAX * FNW + G_MAX) * 4;
  const int recv2_bytes = C == 1 ? 0 : C * (cap2 + 2) * 8;
  // TIP staging: the whole range at once (no refill) with the smallest tile
  // that needs at most ST_MAX_STAGES stages, else a ring of at least two
  // stages holding up to 128 KB.  Warp w scores the 128-token units w,
  // w + W, ...; in a ring, stages x (units per tile) must be a multiple of
  // the W scoring warps so that every warp meets the same stages in every
  // round of ns tiles
  // and so waits on each of their phases in order (a parity wait on a
  // barrier two phases behind would pass at once).
  const int fc_tok = nfc * 2 * ES;  // bytes per token over all planes
  int tile = 0, stages = 0;
  for (int t = TIP_UNIT; t <= 4096 && !tile; t *= 2) {
    const int st = ceil_div(chunkT, t);
    if (st <= ST_MAX_STAGES && st * t * fc_tok <= room) {
      tile = t;
      stages = st;
    }
  }
  int tip_warps = SNW;
  for (int tw = SNW; tw >= FNW && !tile; tw /= 2) {  // fewer scoring warps when no ring aligns for all
    for (int t = 1024; t >= TIP_UNIT && !tile; t /= 2) {
      const int step = std::max(1, tw / (t / TIP_UNIT));  // stage counts that keep the rounds aligned
      int best = 0;
      for (int st = std::max(2, step); st <= ST_MAX_STAGES; st += step) {
        if (st % step != 0) continue;
        if (st * t * fc_tok > std::min(room, std::max(131072, 2 * t * fc_tok))) break;
        best = st;
      }
      if (best) {
        tile = t;
        stages = best;
        tip_warps = tw;
      }
    }
  }
  if (!tile) return FASA_ERR_UNSUPPORTED;
  const int tip_bytes = stages * tile * fc_tok;
  // FAC slots in `big`: two groups in flight per attending warp when they fit
  int wst = 0;
  for (int w = 2; w >= 1 && !wst; --w)
    if (fac_slots(w) + pt_bytes <= room) wst = w;
  if (!wst) return FASA_ERR_UNSUPPORTED;
  // the first-round list is gathered during the exchange when it fits the
  // slots (a longer list streamed after the selection measured slower: the
  // early copies slow the selection and leave fewer slots per warp)
  const int spec = (C > 1 && cap1 <= wst * FNW * GR) ? 1 : 0;
  // Without the first-round gather, every gather follows the selection and
  // its slots start at the histogram: up to FAC_WST_MAX groups in flight per
  // warp over the selection's dead regions and `big`.
  int off_fac = p.off_big, wst_fac = wst;
  if (!spec) {
    off_fac = p.off_hist;
    for (int w = FAC_WST_MAX; w > wst; --w)
      if (off_fac + fac_slots(w) + pt_bytes <= limit) {
        wst_fac = w;
        break;
      }
  }
  // the listed rows' scores, [G_MAX heads][cap1 + 8], beside the slots,
  // then each attending warp's compacted selection (cap1 16-bit entries)
  const int s_bytes = G_MAX * (cap1 + 8) * 4 + align_up((D / 16) * cap1 * 2, 16);
  const int rfac = (spec && fac_slots(wst) + s_bytes <= room) ? 1 : 0;
  const int reload = (s_cap == 0 && !spec && chunkT * 4 <= room) ? 1 : 0;
  int big = std::max(tip_bytes, fac_slots(wst) + (rfac ? std::max(pt_bytes, s_bytes) : pt_bytes));
  big = std::max(big, std::max(rec_bytes, recv2_bytes));
  if (reload) big = std::max(big, chunkT * 4);
  if (big > room) return FASA_ERR_UNSUPPORTED;
  p.s_cap = s_cap;
  p.tip_tile = tile;
  p.tip_stages = stages;
  p.tip_warps = tip_warps;
  p.rho = rho;
  p.cap1 = cap1;
  p.cap2 = cap2;
  p.spec = spec;
  p.rfac = rfac;
  p.fac_wst = wst_fac;
  p.off_fac = off_fac;
  p.rows_cap = rows_cap;
  p.reload = reload;
  p.comb_slot = comb_slot;
  p.comb_sl = sl;
  p.comb_inv_sl = 1.f / (float)sl;
  p.c_magic = div_magic((uint32_t)C);
  p.tt_magic = div_magic((uint32_t)tile);
  // with a first-round gather and at least four warps left over, the union
  // select runs on warps 0..C-1 while the rest gather
  p.u_nuw = (spec && C <= SNW - 4) ? C : SNW;
  p.u_wps = std::max(1, p.u_nuw / C);
  p.u_inv_wps = 1.f / (float)p.u_wps;
  p.off_recv2 = p.off_big;
  p.off_pt = off_fac + fac_slots(wst_fac);
  p.smem_total = std::max(p.off_big + big, p.off_pt + pt_bytes);
  *ws = s_cap == 0 ? (size_t)d->batch * d->n_kv_heads * d->t_max * 4 : 0;
  return FASA_OK;
}

void fill_step(StepParams& p, const fasa_dims_t* d, int32_t budget) {
  memset(&p, 0, sizeof(p));
  p.B = d->batch;
  p.Hq = d->n_q_heads;
  p.Hkv = d->n_kv_heads;
  p.G = d->n_q_heads / d->n_kv_heads;
  p.T_max = d->t_max;
  p.n_tip = d->n_tip;
  p.budget = budget;
  Params tmp;
  fill_rope_turns(tmp, d);
  memcpy(p.rope_turns, tmp.rope_turns, sizeof(p.rope_turns));
  p.wait_ns = g_wait_ns;
  p.drop_stage = g_drop_tip_tile;
  p.drop_refill = g_drop_fac_refill;
}

// The bf16 step kernel serves fasa_decode_step when these dims plan.
bool step_kernel_applies(const fasa_dims_t* d) { return d->dtype == FASA_BF16; }

// Plans (and launches) the step kernel.  Cluster size: the override, else
// the largest C <= 16 for which every unit's cluster is resident at once.
// The kernel serves plans of at least STEP_MIN_C CTAs per unit -- few units
// at small batch, where the step is one latency-bound chain; with fewer,
// larger CTAs (batched or multi-wave shapes) each CTA's lists and row
// gathers are long and the general cluster kernel is faster.
// FASA_ERR_UNSUPPORTED: no plan here; the caller then uses the cluster kernel.
int step_plan_and_launch(StepParams& p, const fasa_dims_t* d, void* ws, size_t ws_bytes, bool launch,
                         size_t* ws_need, int* C_out, cudaStream_t stream) {
  DevInfo di;
  int st = device_info(&di);
  if (st) return st;
  p.status = di.status;
  const int units = d->batch * d->n_kv_heads;
  int C = 0;
  size_t need = 0;
  auto capacity = [&](int c) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, d->head_dim, c, p.smem_total);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const int n = max_active_clusters_step_bf16(d->head_dim, c, p.smem_total);
    cache.emplace(key, n);
    return n;
  };
  if (d->reserved > 0) {
    if (d->reserved < STEP_MIN_C) return FASA_ERR_UNSUPPORTED;
    if (plan_step(p, d, d->reserved, &need, di.smem_optin) != FASA_OK) return FASA_ERR_UNSUPPORTED;
    if (capacity(d->reserved) < 1) return FASA_ERR_UNSUPPORTED;
    C = d->reserved;
  } else {
    for (int c = C_MAX; c >= STEP_MIN_C && !C; --c) {
      if (plan_step(p, d, c, &need, di.smem_optin) != FASA_OK) continue;
      if (capacity(c) >= units) C = c;
    }
    if (!C) return FASA_ERR_UNSUPPORTED;
    if (plan_step(p, d, C, &need, di.smem_optin) != FASA_OK) return FASA_ERR_UNSUPPORTED;
  }
  if (ws_need) *ws_need = need;
  if (C_out) *C_out = C;
  if (!launch) return FASA_OK;
  if (need > 0) {
    if (!ws || ws_bytes < need || !aligned16(ws)) return FASA_ERR_WORKSPACE;
    p.scores = reinterpret_cast<float*>(ws);
  }
  const cudaError_t e = launch_step_bf16(p, d->head_dim, C, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return FASA_OK;
}

// ---------------------------------------------------------------- aux kernels
struct RopeTurns {
  unsigned long long t[64];
};

template <typename T, int D>
__global__ void rope_q_kernel(const T* q, const int* pos, float* q_rot, int Hq, const __grid_constant__ RopeTurns rt) {
  __shared__ float2 cs[D / 2];
  const int b = blockIdx.x;
  const int m = pos[b];
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) cs[i] = rope_cos_sin(rt.t[i], m);
  __syncthreads();
  const T* qb = q + (size_t)b * Hq * D;
  float* ob = q_rot + (size_t)b * Hq * D;
  for (int x = threadIdx.x; x < Hq * (D / 2); x += blockDim.x) {
    const int hq = x / (D / 2), i = x - hq * (D / 2);
    const float x0 = to_f32<T>(qb[hq * D + 2 * i]), x1 = to_f32<T>(qb[hq * D + 2 * i + 1]);
    const float2 c = cs[i];
    ob[hq * D + 2 * i] = x0 * c.x - x1 * c.y;
    ob[hq * D + 2 * i + 1] = x0 * c.y + x1 * c.x;
  }
}

// One FC pair (2 elements) moved as a single word.
template <typename T>
struct Pair;
template <>
struct Pair<float> {
  using type = float2;
};
template <>
struct Pair<__nv_bfloat16> {
  using type = uint32_t;
};

template <typename T>
__global__ void build_kdom_kernel(const T* K, const int* dom, const int* lens, T* kd, int Hkv, int T_max, int D,
                                  int n, int* status) {
  using P = typename Pair<T>::type;
  const int unit = blockIdx.y;
  const int b = unit / Hkv, h = unit - b * Hkv;
  int len = T_max;
  if (lens) {
    len = lens[b];
    if (len < 0 || len > T_max) {
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, 1);
      len = min(max(len, 0), T_max);
    }
  }
  const int tau = blockIdx.x * blockDim.x + threadIdx.x;
  if (tau >= len) return;
  const P* row = reinterpret_cast<const P*>(K + ((size_t)unit * T_max + tau) * D);
  // blocked FC-major layout [unit][tau / KB][j][tau % KB]
  P* dst = reinterpret_cast<P*>(kd) + ((size_t)unit * (T_max / KDOM_BLOCK) + tau / KDOM_BLOCK) * n * KDOM_BLOCK +
           tau % KDOM_BLOCK;
  for (int j = 0; j < n; ++j) {
    int i = dom[h * n + j];
    if (i < 0) continue;  // an unused slot of a head keeping fewer FCs
    if (i >= D / 2) {
      atomicOr(status, 1);
      i = D / 2 - 1;
    }
    dst[(size_t)j * KDOM_BLOCK] = row[i];
  }
}

// K^nondom (FASA-M split keys): per token, the key's FC pairs outside the
// head's dominant set, in FC order: [unit][T_max][d/2 - n] pairs.  A table
// that is not n distinct FCs in range is reported (the layout cannot hold
// it) and its row left unwritten.
template <typename T>
__global__ void build_knondom_kernel(const T* K, const int* dom, const int* lens, T* knd, int Hkv, int T_max, int D,
                                     int n, int* status) {
  using P = typename Pair<T>::type;
  __shared__ uint8_t order[64];  // the non-dominant FCs in order
  __shared__ int ok_s;
  const int unit = blockIdx.y;
  const int b = unit / Hkv, h = unit - b * Hkv;
  const int npairs = D / 2, ndp = npairs - n;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t m0 = 0u, m1 = 0u;
    bool ok = true;
    for (int j = lane; j < n; j += 32) {
      const int i = dom[h * n + j];
      if (i < 0 || i >= npairs) ok = false;
      else if (i < 32) m0 |= 1u << i;
      else m1 |= 1u << (i - 32);
    }
    m0 = __reduce_or_sync(0xffffffffu, m0);
    m1 = __reduce_or_sync(0xffffffffu, m1);
    ok = __all_sync(0xffffffffu, ok) && __popc(m0) + __popc(m1) == n;
    for (int f = lane; f < npairs; f += 32) {
      const bool dm = f < 32 ? ((m0 >> f) & 1u) != 0u : ((m1 >> (f - 32)) & 1u) != 0u;
      if (!dm) {
        const int rank = f < 32 ? __popc(~m0 & ((1u << f) - 1u)) : __popc(~m0) + __popc(~m1 & ((1u << (f - 32)) - 1u));
        if (rank < ndp) order[rank] = (uint8_t)f;
      }
    }
    if (lane == 0) {
      ok_s = ok;
      if (!ok && blockIdx.x == 0) atomicOr(status, 1);
    }
  }
  __syncthreads();
  if (!ok_s) return;
  int len = T_max;
  if (lens) {
    len = lens[b];
    if (len < 0 || len > T_max) {
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, 1);
      len = min(max(len, 0), T_max);
    }
  }
  // thread x: pair x % ndp of token x / ndp of this block's tokens
  const int tok0 = blockIdx.x * 64;
  for (int x = threadIdx.x; x < 64 * ndp; x += blockDim.x) {
    const int tau = tok0 + x / ndp, j = x - (x / ndp) * ndp;
    if (tau >= len) continue;
    const P* row = reinterpret_cast<const P*>(K + ((size_t)unit * T_max + tau) * D);
    reinterpret_cast<P*>(knd)[((size_t)unit * T_max + tau) * ndp + j] = row[order[j]];
  }
}

template <typename T>
__global__ void append_kdom_kernel(const T* k_new, const int* dom, const int* tok_pos, T* kd, int Hkv, int T_max,
                                   int D, int n, int* status) {
  using P = typename Pair<T>::type;
  const int unit = blockIdx.x;
  const int b = unit / Hkv, h = unit - b * Hkv;
  int t = tok_pos[b];
  if (t < 0 || t >= T_max) {
    if (threadIdx.x == 0) atomicOr(status, 1);
    return;
  }
  const P* row = reinterpret_cast<const P*>(k_new + (size_t)unit * D);
  P* dst = reinterpret_cast<P*>(kd) + ((size_t)unit * (T_max / KDOM_BLOCK) + t / KDOM_BLOCK) * n * KDOM_BLOCK +
           t % KDOM_BLOCK;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    int i = dom[h * n + j];
    if (i < 0) continue;  // an unused slot of a head keeping fewer FCs
    if (i >= D / 2) {
      atomicOr(status, 1);
      i = D / 2 - 1;
    }
    dst[(size_t)j * KDOM_BLOCK] = row[i];
  }
}

// fasa_decode_step and fasa_decode_step_split: keys whole in k_cache, or
// (ksplit) their non-dominant pairs there and the dominant ones in k_dom.
int decode_step_impl(const void* q, const int32_t* pos, const void* k_cache, const void* v_cache, const void* k_dom,
                     const int32_t* dom_fc, const int32_t* seq_lens, int32_t budget, float* out, int32_t* idx_out,
                     int32_t* count_out, void* workspace, size_t workspace_bytes, const fasa_dims_t* dims,
                     fasa_stream_t stream, bool ksplit) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q || !pos || !k_cache || !v_cache || !k_dom || !dom_fc || !seq_lens || !out || budget < 1)
    return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_dom) || !aligned16(out)) return FASA_ERR_INVALID_ARG;
  if (ksplit && (dims->dtype != FASA_BF16 || dims->n_tip % 4 != 0)) return FASA_ERR_UNSUPPORTED;
  if (step_kernel_applies(dims)) {
    StepParams sp;
    fill_step(sp, dims, budget);
    sp.q = q;
    sp.pos = pos;
    sp.k_cache = k_cache;
    sp.v_cache = v_cache;
    sp.k_dom = k_dom;
    sp.dom_fc = dom_fc;
    sp.seq_lens = seq_lens;
    sp.out = out;
    sp.idx_out = idx_out;
    sp.count_out = count_out;
    if (ksplit) sp.flags |= F_KSPLIT;
    st = step_plan_and_launch(sp, dims, workspace, workspace_bytes, true, nullptr, nullptr,
                              reinterpret_cast<cudaStream_t>(stream));
    if (st != FASA_ERR_UNSUPPORTED) return st;
  }
  Params p;
  fill_common(p, dims, budget, nullptr);
  p.q = q;
  p.pos = pos;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_dom = k_dom;
  p.dom_fc = dom_fc;
  p.seq_lens = seq_lens;
  p.out = out;
  p.idx_out = idx_out;
  p.count_out = count_out;
  int flags = F_ROPE | F_TIP | F_SELECT | F_FAC;
  if (idx_out || count_out) flags |= F_IDX_OUT;
  if (ksplit) flags |= F_KSPLIT;
  return plan_and_launch(p, dims, flags, workspace, workspace_bytes, true, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

// fasa_decode_step_append and its split-key form (ksplit: k_cache holds the
// keys' non-dominant pairs; the new token's are written there).
int decode_append_impl(const void* q, const void* k_new, const void* v_new, const int32_t* seq_lens, void* k_cache,
                       void* v_cache, void* k_dom, const int32_t* dom_fc, int32_t budget, float* out,
                       int32_t* idx_out, int32_t* count_out, void* workspace, size_t workspace_bytes,
                       const fasa_dims_t* dims, fasa_stream_t stream, bool ksplit) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !k_dom || !dom_fc || !seq_lens || !out || budget < 1)
    return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_dom) || !aligned16(out)) return FASA_ERR_INVALID_ARG;
  if (ksplit && (dims->dtype != FASA_BF16 || dims->n_tip % 4 != 0)) return FASA_ERR_UNSUPPORTED;
  if (step_kernel_applies(dims)) {
    StepParams sp;
    fill_step(sp, dims, budget);
    sp.flags = F_APPEND | (ksplit ? F_KSPLIT : 0);
    sp.q = q;
    sp.pos = seq_lens;
    sp.k_new = k_new;
    sp.v_new = v_new;
    sp.k_cache = k_cache;
    sp.v_cache = v_cache;
    sp.k_dom = k_dom;
    sp.dom_fc = dom_fc;
    sp.seq_lens = seq_lens;
    sp.out = out;
    sp.idx_out = idx_out;
    sp.count_out = count_out;
    st = step_plan_and_launch(sp, dims, workspace, workspace_bytes, true, nullptr, nullptr,
                              reinterpret_cast<cudaStream_t>(stream));
    if (st != FASA_ERR_UNSUPPORTED) return st;
  }
  Params p;
  fill_common(p, dims, budget, nullptr);
  p.q = q;
  p.pos = seq_lens;  // the query sits at the new token's position, len
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_dom = k_dom;
  p.dom_fc = dom_fc;
  p.seq_lens = seq_lens;
  p.out = out;
  p.idx_out = idx_out;
  p.count_out = count_out;
  int flags = F_ROPE | F_TIP | F_SELECT | F_FAC | F_APPEND;
  if (idx_out || count_out) flags |= F_IDX_OUT;
  if (ksplit) flags |= F_KSPLIT;
  return plan_and_launch(p, dims, flags, workspace, workspace_bytes, true, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

// ============================================================================
extern "C" {

int fasa_version(void) { return 100; }

const char* fasa_status_string(int status) {
  switch (status) {
    case FASA_OK: return "FASA_OK";
    case FASA_ERR_INVALID_ARG: return "FASA_ERR_INVALID_ARG";
    case FASA_ERR_UNSUPPORTED: return "FASA_ERR_UNSUPPORTED";
    case FASA_ERR_WORKSPACE: return "FASA_ERR_WORKSPACE";
    case FASA_ERR_CUDA: return "FASA_ERR_CUDA";
    default: return "FASA_ERR_UNKNOWN";
  }
}

int fasa_last_cuda_error(void) { return t_last_cuda_error; }

int fasa_max_budget(const fasa_dims_t* dims, int32_t* max_budget) {
  int st = check_dims(dims);
  if (st) return st;
  if (!max_budget) return FASA_ERR_INVALID_ARG;
  DevInfo di;
  st = device_info(&di);
  if (st) return st;
  // the fused step has the tightest shared-memory plan; search its limit
  int lo = 0, hi = 1 << 20;
  const int flags = F_ROPE | F_TIP | F_SELECT | F_FAC | F_IDX_OUT;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    Params p;
    fill_common(p, dims, mid, di.status);
    size_t ws = 0;
    bool ok = false;
    for (int C = dims->reserved > 0 ? dims->reserved : C_MAX; C >= 1; --C) {
      if (plan_smem(p, dims, C, flags, true, &ws, di.smem_optin) == FASA_OK) {
        ok = true;
        break;
      }
      if (dims->reserved > 0) break;
    }
    if (ok) lo = mid;
    else hi = mid - 1;
  }
  *max_budget = lo;
  return FASA_OK;
}

int fasa_workspace_size(const fasa_dims_t* dims, int32_t budget, size_t* bytes) {
  int st = check_dims(dims);
  if (st) return st;
  if (!bytes || budget < 1) return FASA_ERR_INVALID_ARG;
  if (step_kernel_applies(dims)) {
    StepParams sp;
    fill_step(sp, dims, budget);
    st = step_plan_and_launch(sp, dims, nullptr, 0, false, bytes, nullptr, nullptr);
    if (st != FASA_ERR_UNSUPPORTED) return st;
  }
  Params p;
  fill_common(p, dims, budget, nullptr);
  return plan_and_launch(p, dims, F_ROPE | F_TIP | F_SELECT | F_FAC | F_IDX_OUT, nullptr, 0, false, bytes, nullptr,
                         nullptr);
}

int fasa_cluster_size(const fasa_dims_t* dims, int32_t* ctas) {
  int st = check_dims(dims);
  if (st) return st;
  if (!ctas) return FASA_ERR_INVALID_ARG;
  int C = 0;
  if (step_kernel_applies(dims)) {
    StepParams sp;
    fill_step(sp, dims, 1);
    st = step_plan_and_launch(sp, dims, nullptr, 0, false, nullptr, &C, nullptr);
    if (st == FASA_OK) {
      *ctas = C;
      return FASA_OK;
    }
    if (st != FASA_ERR_UNSUPPORTED) return st;
  }
  Params p;
  fill_common(p, dims, 1, nullptr);
  st = plan_and_launch(p, dims, F_ROPE | F_TIP | F_SELECT | F_FAC | F_IDX_OUT, nullptr, 0, false, nullptr, &C,
                       nullptr);
  if (st) return st;
  *ctas = C;
  return FASA_OK;
}

int fasa_step_kernel(const fasa_dims_t* dims, int32_t* kernel) {
  int st = check_dims(dims);
  if (st) return st;
  if (!kernel) return FASA_ERR_INVALID_ARG;
  *kernel = FASA_KERNEL_CLUSTER;
  if (step_kernel_applies(dims)) {
    StepParams sp;
    fill_step(sp, dims, 1);
    int C = 0;
    st = step_plan_and_launch(sp, dims, nullptr, 0, false, nullptr, &C, nullptr);
    if (st == FASA_OK) *kernel = FASA_KERNEL_SINGLE_EXCHANGE;
    else if (st != FASA_ERR_UNSUPPORTED) return st;
  }
  return FASA_OK;
}

int fasa_apply_rope_q(const void* q, const int32_t* pos, float* q_rot, const fasa_dims_t* dims,
                      fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q || !pos || !q_rot) return FASA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int D = dims->head_dim;
  const dim3 grid(dims->batch);
  const int Hq = dims->n_q_heads;
  Params tmp;
  fill_rope_turns(tmp, dims);
  RopeTurns rt;
  memcpy(rt.t, tmp.rope_turns, sizeof(rt.t));
  if (dims->dtype == FASA_F32) {
    if (D == 128) rope_q_kernel<float, 128><<<grid, 256, 0, s>>>((const float*)q, pos, q_rot, Hq, rt);
    else rope_q_kernel<float, 64><<<grid, 256, 0, s>>>((const float*)q, pos, q_rot, Hq, rt);
  } else {
    using B16 = __nv_bfloat16;
    if (D == 128) rope_q_kernel<B16, 128><<<grid, 256, 0, s>>>((const B16*)q, pos, q_rot, Hq, rt);
    else rope_q_kernel<B16, 64><<<grid, 256, 0, s>>>((const B16*)q, pos, q_rot, Hq, rt);
  }
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FASA_OK : cuda_fail(e);
}

int fasa_build_kdom(const void* k_cache, const int32_t* dom_fc, const int32_t* seq_lens, void* k_dom,
                    const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!k_cache || !dom_fc || !k_dom) return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(k_dom)) return FASA_ERR_INVALID_ARG;
  DevInfo di;
  st = device_info(&di);
  if (st) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(ceil_div(dims->t_max, 256), dims->batch * dims->n_kv_heads);
  if (dims->dtype == FASA_F32)
    build_kdom_kernel<float><<<grid, 256, 0, s>>>((const float*)k_cache, dom_fc, seq_lens, (float*)k_dom,
                                                  dims->n_kv_heads, dims->t_max, dims->head_dim, dims->n_tip,
                                                  di.status);
  else
    build_kdom_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)k_cache, dom_fc, seq_lens,
                                                          (__nv_bfloat16*)k_dom, dims->n_kv_heads, dims->t_max,
                                                          dims->head_dim, dims->n_tip, di.status);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FASA_OK : cuda_fail(e);
}

int fasa_build_knondom(const void* k_cache, const int32_t* dom_fc, const int32_t* seq_lens, void* k_nondom,
                       const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!k_cache || !dom_fc || !k_nondom) return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(k_nondom)) return FASA_ERR_INVALID_ARG;
  if (dims->n_tip >= dims->head_dim / 2) return FASA_OK;  // no non-dominant pairs
  DevInfo di;
  st = device_info(&di);
  if (st) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(ceil_div(dims->t_max, 64), dims->batch * dims->n_kv_heads);
  if (dims->dtype == FASA_F32)
    build_knondom_kernel<float><<<grid, 256, 0, s>>>((const float*)k_cache, dom_fc, seq_lens, (float*)k_nondom,
                                                     dims->n_kv_heads, dims->t_max, dims->head_dim, dims->n_tip,
                                                     di.status);
  else
    build_knondom_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)k_cache, dom_fc, seq_lens,
                                                             (__nv_bfloat16*)k_nondom, dims->n_kv_heads,
                                                             dims->t_max, dims->head_dim, dims->n_tip, di.status);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FASA_OK : cuda_fail(e);
}

int fasa_append_kdom(const void* k_new, const int32_t* dom_fc, const int32_t* tok_pos, void* k_dom,
                     const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!k_new || !dom_fc || !tok_pos || !k_dom) return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_dom)) return FASA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) & (uintptr_t)(2 * elem_size(dims) - 1)) != 0) return FASA_ERR_INVALID_ARG;
  DevInfo di;
  st = device_info(&di);
  if (st) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(dims->batch * dims->n_kv_heads);
  const int threads = dims->n_tip < 32 ? 32 : 64;
  if (dims->dtype == FASA_F32)
    append_kdom_kernel<float><<<grid, threads, 0, s>>>((const float*)k_new, dom_fc, tok_pos, (float*)k_dom,
                                                       dims->n_kv_heads, dims->t_max, dims->head_dim, dims->n_tip,
                                                       di.status);
  else
    append_kdom_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>((const __nv_bfloat16*)k_new, dom_fc, tok_pos,
                                                               (__nv_bfloat16*)k_dom, dims->n_kv_heads,
                                                               dims->t_max, dims->head_dim, dims->n_tip, di.status);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FASA_OK : cuda_fail(e);
}

int fasa_tip_score(const float* q_rot, const void* k_dom, const int32_t* dom_fc, const int32_t* seq_lens,
                   float* scores, const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q_rot || !k_dom || !dom_fc || !seq_lens || !scores) return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_dom) || !aligned16(scores) || !aligned16(q_rot)) return FASA_ERR_INVALID_ARG;
  Params p;
  fill_common(p, dims, 1, nullptr);
  p.q_rot = q_rot;
  p.k_dom = k_dom;
  p.dom_fc = dom_fc;
  p.seq_lens = seq_lens;
  p.scores = scores;
  return plan_and_launch(p, dims, F_TIP, nullptr, 0, true, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int fasa_topk_select(const float* scores, const int32_t* seq_lens, int32_t budget, int32_t* idx, int32_t* count,
                     const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!scores || !seq_lens || !idx || !count || budget < 1) return FASA_ERR_INVALID_ARG;
  if (!aligned16(scores)) return FASA_ERR_INVALID_ARG;
  Params p;
  fill_common(p, dims, budget, nullptr);
  p.scores_in = scores;
  p.seq_lens = seq_lens;
  p.idx_out = idx;
  p.count_out = count;
  return plan_and_launch(p, dims, F_SC_IN | F_SELECT | F_IDX_OUT, nullptr, 0, true, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

int fasa_focused_attention(const float* q_rot, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                           const int32_t* idx, const int32_t* count, int32_t budget, float* out,
                           const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q_rot || !k_cache || !v_cache || !seq_lens || !idx || !count || !out || budget < 1)
    return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q_rot) || !aligned16(out)) return FASA_ERR_INVALID_ARG;
  Params p;
  fill_common(p, dims, budget, nullptr);
  p.q_rot = q_rot;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.seq_lens = seq_lens;
  p.idx_in = idx;
  p.count_in = count;
  p.out = out;
  return plan_and_launch(p, dims, F_FAC | F_IDX_IN, nullptr, 0, true, nullptr, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

int fasa_dense_attention(const float* q_rot, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                         float* out, const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q_rot || !k_cache || !v_cache || !seq_lens || !out) return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q_rot) || !aligned16(out)) return FASA_ERR_INVALID_ARG;
  Params p;
  fill_common(p, dims, 1, nullptr);
  p.q_rot = q_rot;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.seq_lens = seq_lens;
  p.out = out;
  return plan_and_launch(p, dims, F_DENSE, nullptr, 0, true, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int fasa_decode_step(const void* q, const int32_t* pos, const void* k_cache, const void* v_cache, const void* k_dom,
                     const int32_t* dom_fc, const int32_t* seq_lens, int32_t budget, float* out, int32_t* idx_out,
                     int32_t* count_out, void* workspace, size_t workspace_bytes, const fasa_dims_t* dims,
                     fasa_stream_t stream) {
  return decode_step_impl(q, pos, k_cache, v_cache, k_dom, dom_fc, seq_lens, budget, out, idx_out, count_out,
                          workspace, workspace_bytes, dims, stream, false);
}

int fasa_decode_step_split(const void* q, const int32_t* pos, const void* k_nondom, const void* v_cache,
                           const void* k_dom, const int32_t* dom_fc, const int32_t* seq_lens, int32_t budget,
                           float* out, int32_t* idx_out, int32_t* count_out, void* workspace, size_t workspace_bytes,
                           const fasa_dims_t* dims, fasa_stream_t stream) {
  return decode_step_impl(q, pos, k_nondom, v_cache, k_dom, dom_fc, seq_lens, budget, out, idx_out, count_out,
                          workspace, workspace_bytes, dims, stream, true);
}

int fasa_decode_step_append(const void* q, const void* k_new, const void* v_new, const int32_t* seq_lens,
                            void* k_cache, void* v_cache, void* k_dom, const int32_t* dom_fc, int32_t budget,
                            float* out, int32_t* idx_out, int32_t* count_out, void* workspace,
                            size_t workspace_bytes, const fasa_dims_t* dims, fasa_stream_t stream) {
  return decode_append_impl(q, k_new, v_new, seq_lens, k_cache, v_cache, k_dom, dom_fc, budget, out, idx_out,
                            count_out, workspace, workspace_bytes, dims, stream, false);
}

int fasa_decode_step_append_split(const void* q, const void* k_new, const void* v_new, const int32_t* seq_lens,
                                  void* k_nondom, void* v_cache, void* k_dom, const int32_t* dom_fc, int32_t budget,
                                  float* out, int32_t* idx_out, int32_t* count_out, void* workspace,
                                  size_t workspace_bytes, const fasa_dims_t* dims, fasa_stream_t stream) {
  return decode_append_impl(q, k_new, v_new, seq_lens, k_nondom, v_cache, k_dom, dom_fc, budget, out, idx_out,
                            count_out, workspace, workspace_bytes, dims, stream, true);
}

int fasa_fc_agreement_workspace_size(const fasa_dims_t* dims, size_t* bytes) {
  if (!bytes) return FASA_ERR_INVALID_ARG;
  *bytes = 0;
  const int st = check_dims(dims);
  if (st) return st;
  *bytes = fc_agreement_workspace(dims->batch * dims->n_kv_heads, dims->head_dim, dims->t_max);
  return FASA_OK;
}

int fasa_fc_agreement(const float* q_rot, const void* k_cache, const int32_t* seq_lens, int32_t topk, float* ca,
                      void* workspace, size_t workspace_bytes, const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q_rot || !k_cache || !seq_lens || !ca || topk < 1) return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(q_rot)) return FASA_ERR_INVALID_ARG;
  const size_t need = fc_agreement_workspace(dims->batch * dims->n_kv_heads, dims->head_dim, dims->t_max);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FASA_ERR_WORKSPACE;
  DevInfo di;
  st = device_info(&di);
  if (st) return st;
  const cudaError_t e = launch_fc_agreement(q_rot, k_cache, seq_lens, nullptr, 0, topk, ca, dims->batch,
                                            dims->n_q_heads, dims->n_kv_heads, dims->head_dim, dims->t_max,
                                            dims->dtype == FASA_BF16, workspace, di.status,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FASA_OK : cuda_fail(e);
}

int fasa_compound_agreement(const float* q_rot, const void* k_cache, const int32_t* dom_fc,
                            const int32_t* seq_lens, int32_t topk, float* cca, void* workspace,
                            size_t workspace_bytes, const fasa_dims_t* dims, fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!q_rot || !k_cache || !dom_fc || !seq_lens || !cca || topk < 1) return FASA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(q_rot)) return FASA_ERR_INVALID_ARG;
  const size_t need = fc_agreement_workspace(dims->batch * dims->n_kv_heads, dims->head_dim, dims->t_max);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FASA_ERR_WORKSPACE;
  DevInfo di;
  st = device_info(&di);
  if (st) return st;
  const cudaError_t e = launch_fc_agreement(q_rot, k_cache, seq_lens, dom_fc, dims->n_tip, topk, cca, dims->batch,
                                            dims->n_q_heads, dims->n_kv_heads, dims->head_dim, dims->t_max,
                                            dims->dtype == FASA_BF16, workspace, di.status,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FASA_OK : cuda_fail(e);
}

int fasa_select_dominant_fcs(const float* ca_mean, int32_t n_tip, int32_t* dom_fc, const fasa_dims_t* dims,
                             fasa_stream_t stream) {
  int st = check_dims(dims);
  if (st) return st;
  if (!ca_mean || !dom_fc || n_tip < 1 || n_tip > dims->head_dim / 2) return FASA_ERR_INVALID_ARG;
  const cudaError_t e = launch_select_dominant(ca_mean, dims->n_kv_heads, dims->head_dim / 2, n_tip, dom_fc,
                                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FASA_OK : cuda_fail(e);
}


int fasa_test_fault_injection(uint64_t wait_limit_ns, int32_t drop_tip_tile, int32_t drop_fac_refill) {
  if (wait_limit_ns == 0 || drop_tip_tile < -1 || drop_fac_refill < -1) return FASA_ERR_INVALID_ARG;
  g_wait_ns = wait_limit_ns;
  g_drop_tip_tile = drop_tip_tile;
  g_drop_fac_refill = drop_fac_refill;
  return FASA_OK;
}

int fasa_device_status(fasa_stream_t stream, int32_t* status) {
  if (!status) return FASA_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  *status = v;
  return FASA_OK;
}

}  // extern "C"
