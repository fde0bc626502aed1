// Internal definitions shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fasa {

constexpr int NT = 256;          // threads per CTA of the cluster kernel
constexpr int NW = NT / 32;      // warps per CTA
constexpr int RT = 32;           // FAC rows per pipeline tile (fp32 path)
constexpr int FAC_STAGES = 4;    // cp.async ring depth of the FAC gather (fp32 path)
constexpr int GR = 16;           // FAC rows per warp group (bf16 tensor-core path)
constexpr int PTS = 24;          // row stride (floats) of a warp's softmax-weight tile
constexpr int G_MAX = 8;         // largest GQA group
constexpr int C_MAX = 16;        // largest cluster
constexpr int KDOM_BLOCK = 64;   // tokens per block of the dominant-key copy
constexpr int MISC_BYTES = 512;  // broadcast / reduction scratch in shared memory
// Radix digits of the 32-bit score keys: 12 + 10 + 10 bits.
constexpr int HLOC_BINS = 4096;  // local histogram (largest digit)
constexpr int HLEAD_BINS = 4096 + 1024 + 1024;  // cluster totals of the three digits

// What one launch of the cluster kernel does.
enum : int {
  F_ROPE = 1 << 0,     // q is the pre-RoPE stored query: rotate in the kernel
  F_TIP = 1 << 1,      // compute TIP scores from k_dom
  F_SC_IN = 1 << 2,    // take scores from p.scores_in instead
  F_SELECT = 1 << 3,   // top-k selection
  F_IDX_OUT = 1 << 4,  // write idx / count
  F_FAC = 1 << 5,      // attention over the selected rows
  F_IDX_IN = 1 << 6,   // selected rows come from p.idx_in / p.count_in
  F_DENSE = 1 << 7,    // attention over every cached row
  F_APPEND = 1 << 8,   // step: first append the new token (k_new, v_new) at index len
  F_KSPLIT = 1 << 9,   // keys in two parts (FASA-M): k_cache holds each token's non-dominant
                       // FC pairs (row of d - 2 n_tip elements), k_dom the dominant ones
};

struct Params {
  int B, Hq, Hkv, G, T_max, n_tip, budget, flags;
  // RoPE frequencies as fixed-point turns: rope_turns[i] = theta_i / (2 pi) * 2^64
  // (theta_i = B^(-2i/d)); pos * rope_turns[i] mod 2^64 is the angle in turns.
  unsigned long long rope_turns[64];
  const void* q;            // pre-RoPE stored query (F_ROPE)
  const float* q_rot;       // rotated fp32 query (otherwise)
  const int* pos;
  const void* k_cache;
  const void* v_cache;
  const void* k_dom;
  const int* dom_fc;
  const int* seq_lens;
  const float* scores_in;   // F_SC_IN
  float* scores;            // TIP output (s_cap == 0) -- global [B,Hkv,T_max]
  const void* k_new;        // F_APPEND: the new token's pre-RoPE key [B,Hkv,d]
  const void* v_new;        //           and value [B,Hkv,d]
  const int* idx_in;        // F_IDX_IN
  const int* count_in;
  int* idx_out;             // F_IDX_OUT
  int* count_out;
  float* out;               // [B,Hq,D] fp32
  int* status;              // device status word
  unsigned long long wait_ns;  // bound of every device wait
  int drop_stage;           // test hook: this TIP tile's copy is never issued (-1: none)
  // shared-memory layout (bytes), computed by the host
  int s_cap;                // scores kept per CTA in shared memory (0: global)
  int tip_tile;             // tokens per TIP pipeline tile
  int tip_stages;           // TIP ring depth
  int cand_cap;             // candidate entries per CTA
  int idx_cap;              // selected-index entries per CTA
  int hpc;                  // heads combined per CTA = ceil(G / C)
  int fac_off;              // byte offset of the FAC staging ring inside the big region
  int fac_wst;              // bf16 FAC: groups in flight per warp (1 or 2)
  int off_bar, off_misc, off_qrot, off_qbar, off_stile, off_hloc, off_hlead, off_sc, off_idx, off_own,
      off_part, off_recv, off_big, smem_total;
};

// The bf16 fused-step kernel (fasa_step.cuh): its plan and arguments.
constexpr int SNT = 512;           // threads of a step CTA
constexpr int SNW = SNT / 32;      // its warps
constexpr int FNW = 8;             // warps that attend rows (one 16-row group slot set each)
constexpr int FAC_WST_MAX = 4;     // FAC groups in flight per attending warp, at most
constexpr int ST_MAX_STAGES = 12;  // TIP stage mbarriers [0, 12)
constexpr int ST_BARS = 16;        // + two selection exchanges, the combine, the score reload
constexpr int ST_MISC_BYTES = 1152;
constexpr int UH_BINS = 256;       // histogram of the union's 8-bit digits
constexpr int TIP_UNIT = 128;      // tokens per warp step of TIP (32 lanes x 4)

struct StepParams {
  int B, Hq, Hkv, G, T_max, n_tip, budget, flags;
  // RoPE frequencies as fixed-point turns: theta_i / (2 pi) * 2^64
  unsigned long long rope_turns[64];
  const void* q;  // pre-RoPE stored query [B, Hq, D]
  const int* pos;
  const void* k_cache;
  const void* v_cache;
  const void* k_dom;
  const int* dom_fc;
  const int* seq_lens;
  float* scores;  // [B, Hkv, T_max] score workspace when s_cap == 0
  const void* k_new;  // F_APPEND: the new token's pre-RoPE key [B, Hkv, D]
  const void* v_new;  //           and value [B, Hkv, D]
  int* idx_out;
  int* count_out;
  float* out;
  int* status;
  unsigned long long wait_ns; // bound of every device wait
  int drop_stage;             // test hook: this TIP tile's copy is never issued (-1: none)
  int drop_refill;            // test hook: this refill of attending warp 0's slots is never
                              // reported complete (-1: none)
  // plan (host)
  int s_cap;       // scores per CTA kept in shared memory (0: workspace)
  int tip_tile;    // tokens per TIP stage (multiple of TIP_UNIT)
  int tip_stages;  // TIP ring depth (>= the CTA's tiles: no refill)
  int tip_warps;   // warps that score TIP units (SNW, or 8 for some rings)
  int rho;         // first-round list length per CTA
  int cap1, cap2;  // receive slots per source CTA, first and second round
  int spec;        // gather the first-round list before the selection is final
  int rfac;        // spec, and the listed rows' scores fit beside the resident slots:
                   // the scores are taken during the selection, the FAC after it
                   // splits the head dims over warps (no per-warp records)
  int fac_wst;     // FAC groups in flight per warp (1 .. FAC_WST_MAX)
  int off_fac;     // the FAC group slots: `big`, or (no first-round gather) the
                   // histogram onwards, the selection's regions being dead by then
  int rows_cap;    // capacity of the own-selection list
  int reload;      // copy workspace scores back into shared memory for the sweeps
  int comb_slot;   // bytes of one combine slot: an output slice and every head's (m, l)
  int comb_sl;     // float4 groups of the output per slice (ceil(G D / 4 / C))
  float comb_inv_sl;  // 1 / comb_sl (rounded)
  // divisions by the cluster size and the TIP tile as a multiply-high by
  // floor(2^32 / divisor) (0xffffffff for 1) and one correction step
  uint32_t c_magic, tt_magic;
  // the union select: warps taking part, and warps per source list
  int u_nuw, u_wps;
  float u_inv_wps;
  int off_bar, off_fbar, off_misc, off_qrot, off_qbar, off_hist, off_uh, off_sc, off_recv1, off_rows, off_comb,
      off_comb_snd, off_big, off_recv2, off_pt, smem_total;
};

// Kernel launchers (one translation unit per storage type).
cudaError_t launch_cluster_bf16(const Params& p, int head_dim, int C, cudaStream_t s);
cudaError_t launch_cluster_f32(const Params& p, int head_dim, int C, cudaStream_t s);
// Prepares function attributes and returns the number of co-resident clusters
// of size C for this configuration (0 if C cannot be launched).
int max_active_clusters_bf16(int flags, int head_dim, int C, int smem_bytes);
int max_active_clusters_f32(int flags, int head_dim, int C, int smem_bytes);
cudaError_t launch_step_bf16(const StepParams& p, int head_dim, int C, cudaStream_t s);
int max_active_clusters_step_bf16(int head_dim, int C, int smem_bytes);

// Contextual Agreement and the choice of dominant FCs (fasa_ca.cu).
size_t fc_agreement_workspace(int units, int D, int T_max);
// dom_fc null: the CA of every FC (ca [B*Hkv, D/2]); else the compound CA of
// the n_tip FCs dom_fc[h, :] (ca [B*Hkv]).
cudaError_t launch_fc_agreement(const float* q_rot, const void* k, const int* lens, const int* dom_fc, int n_tip,
                                int K, float* ca, int B, int Hq, int Hkv, int D, int T_max, bool bf16, void* ws,
                                int* status, cudaStream_t s);
cudaError_t launch_select_dominant(const float* ca_mean, int Hkv, int F, int n, int* dom_fc, cudaStream_t s);

}  // namespace fasa
