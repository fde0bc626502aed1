/*
 * fasa.h -- C ABI of the FASA decode-step library (libfasa.so, sm_103a).
 *
 * FASA ("FASA: Frequency-aware Sparse Attention") splits one decode step of
 * attention into Token Importance Prediction (TIP), a per-(batch, KV head)
 * top-k, and Focused Attention Computation (FAC).  The functions below are
 * those stages, a fused step, a dense baseline built from the same kernels,
 * and the maintenance of the dominant-key side copy the TIP stage reads.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is owned by the caller and is a DEVICE pointer
 *    unless one of the two placements below says otherwise.  Nothing is
 *    allocated or freed by the library.  Calls are asynchronous on
 *    `stream` (NULL = the legacy default stream).
 *  - FASA-M placement (the FASA pages, "Hardware-Aware Variants": keep the
 *    dominant key cache on the GPU, offload the rest of the KV cache to host
 *    memory and move only the selected tokens): k_cache and v_cache of
 *    fasa_decode_step, fasa_decode_step_append, fasa_decode_step_noalloc,
 *    fasa_focused_attention and fasa_dense_attention may instead point to
 *    page-locked host memory that the device can address (cudaHostAlloc /
 *    cudaHostRegister, same pointer on the device).  Those entry points read
 *    the caches only row by row in the attention gather (and the append step
 *    writes its one row), so a step then moves just the selected K/V rows
 *    over the host link; TIP reads k_dom, which stays in device memory.
 *  - Zero-copy step I/O: the per-step inputs and outputs of fasa_decode_step
 *    (q, pos, seq_lens, out, idx_out, count_out) may also be page-locked
 *    host memory addressable by the device.  The kernel reads them (a few
 *    KB) and writes them in place over the host link, so a host-driven
 *    decode loop needs no separate copies around the step; the caller
 *    synchronises the stream before reading the results.
 *  - Return value: FASA_OK, or an error code.  Arguments are validated on
 *    the host before any launch; on an error nothing is launched and nothing
 *    is written.  Values that live in device memory (sequence lengths,
 *    positions, FC indices, index lists) cannot be checked on the host: the
 *    kernels clamp them into range and raise FASA_DEV_BAD_INPUT in the device
 *    status word (see fasa_device_status).
 *  - Shapes (row-major, contiguous):
 *      q         [B, Hq, d]            storage dtype, pre-RoPE query
 *      q_rot     [B, Hq, d]            fp32, rotated query
 *      pos       [B]                   int32, query position (usually = len)
 *      k_cache   [B, Hkv, T_max, d]    storage dtype, keys AFTER RoPE
 *      v_cache   [B, Hkv, T_max, d]    storage dtype
 *      k_dom     [B, Hkv, T_max/64, n_tip, 64, 2]  storage dtype: the
 *                                      dominant key columns, FC-major within
 *                                      blocks of 64 tokens
 *      dom_fc    [Hkv, n_tip]          int32, dominant FC indices in [0, d/2);
 *                                      a negative entry marks an unused
 *                                      slot: head h's set I_dom is its
 *                                      entries before the first negative one
 *                                      (at least one), so heads may keep
 *                                      different numbers of FCs (the per-head
 *                                      N_tip of the FASA pages' "Layer-wise
 *                                      and head-wise N_tip optimization").
 *                                      n_tip is the longest set; a head with
 *                                      fewer FCs reads only its planes.
 *      seq_lens  [B]                   int32, cached tokens 0..len-1
 *      scores    [B, Hkv, T_max]       fp32 (entries tau >= len unspecified)
 *      idx       [B, Hkv, budget]      int32, ascending; -1 past count
 *      count     [B, Hkv]              int32, = min(budget, len)
 *      out       [B, Hq, d]            fp32
 *    Query head hq belongs to KV head hq / G, G = Hq / Hkv.
 *  - Frequency chunk (FC) i is the interleaved pair of dimensions (2i, 2i+1).
 *  - Alignment: k_cache, v_cache, k_dom, scores, q_rot and out must be
 *    16-byte aligned; T_max must be a multiple of 64.
 *  - Supported: dtype FASA_F32 or FASA_BF16 (q, caches and k_dom share it),
 *    head_dim 64 or 128, 1 <= G <= 8, 1 <= budget <= fasa_max_budget().
 */
#ifndef FASA_H_
#define FASA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* fasa_stream_t;

/* Host-side status codes. */
enum {
  FASA_OK = 0,
  FASA_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, misalignment, bad budget */
  FASA_ERR_UNSUPPORTED = 2,  /* dtype / head_dim / group size not compiled in   */
  FASA_ERR_WORKSPACE = 3,    /* workspace missing or too small                  */
  FASA_ERR_CUDA = 4          /* a CUDA call failed; see fasa_last_cuda_error()  */
};

/* Device status word bits (fasa_device_status). */
enum {
  FASA_DEV_BAD_INPUT = 1,    /* a device-resident value was out of range and clamped */
  FASA_DEV_TIMEOUT = 2,      /* a bounded device wait expired (a copy or a peer CTA) */
  FASA_DEV_UNDRAINED = 4     /* after a timeout a copy had still not landed: the     */
                             /* kernel left its staging memory alone and skipped the */
                             /* attention of the affected rows (outputs unreliable)  */
};

enum { FASA_F32 = 0, FASA_BF16 = 1 };

typedef struct fasa_dims {
  int32_t batch;       /* B                                   */
  int32_t n_q_heads;   /* Hq                                  */
  int32_t n_kv_heads;  /* Hkv (Hq % Hkv == 0)                 */
  int32_t head_dim;    /* d: 64 or 128                        */
  int32_t t_max;       /* cache capacity per (b, KV head)     */
  int32_t n_tip;       /* dominant FCs per KV head, 1..d/2    */
  int32_t dtype;       /* FASA_F32 or FASA_BF16               */
  int32_t reserved;    /* 0, or a cluster size 1..16 to force  */
  double rope_theta;   /* RoPE base B: theta_i = B^(-2i/d)    */
} fasa_dims_t;

/* Library version (major * 10000 + minor * 100 + patch). */
int fasa_version(void);

/* Human-readable name of a status code (static string). */
const char* fasa_status_string(int status);

/* The cudaError_t of the last call that returned FASA_ERR_CUDA. */
int fasa_last_cuda_error(void);

/* Largest budget (N_fac) the selection kernels accept for these dims. */
int fasa_max_budget(const fasa_dims_t* dims, int32_t* max_budget);

/*
 * Workspace bytes fasa_decode_step needs for these dims and budget (0 when
 * every intermediate fits in on-chip shared memory, which holds for T_max up
 * to 131072).  The workspace is device memory owned by the caller.
 */
int fasa_workspace_size(const fasa_dims_t* dims, int32_t budget, size_t* bytes);

/*
 * RoPE of the query ("FASA: Frequency-aware Sparse Attention", §3.4 "RoPE from
 * a Frequency-Chunk Perspective": theta_i = B^(-2i/d); each FC is turned by the
 * 2x2 rotation R_{m,theta_i}, m = pos[b]).  q_rot = R(pos) q, fp32.
 * The angle m * theta_i is formed exactly in 64-bit fixed-point turns
 * (theta_i / 2pi tabulated from a double-precision pow), so its error does not
 * grow with the position; cos/sin are evaluated in fp32.
 */
int fasa_apply_rope_q(const void* q, const int32_t* pos, float* q_rot,
                      const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * Builds the dominant key cache C_key^dom (same page, "Hardware-Aware Variants",
 * FASA-M/FASA-C: t x d_dom per head, d_dom = 2 N_tip), FC-major within blocks
 * of 64 tokens: k_dom[b,h,tau/64,j,tau%64,0:2] =
 * k_cache[b,h,tau, 2*dom_fc[h,j] : 2*dom_fc[h,j]+2] for tau < seq_lens[b]
 * (all tau < T_max when seq_lens is NULL).  A pure copy; one tile of whole
 * blocks is one contiguous range, so the TIP stage moves it with one bulk copy
 * (a head keeping fewer FCs: one copy of its leading planes per block).
 * Unused slots (negative entries) are left untouched.
 */
int fasa_build_kdom(const void* k_cache, const int32_t* dom_fc, const int32_t* seq_lens,
                    void* k_dom, const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * Appends one token per sequence to k_dom: k_new [B, Hkv, d] holds the new
 * post-RoPE keys, tok_pos [B] their cache slots (< T_max).
 */
int fasa_append_kdom(const void* k_new, const int32_t* dom_fc, const int32_t* tok_pos,
                     void* k_dom, const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * TIP (same page, §3.4 "Online Stage 1: Token Importance Predictor"): for
 * every cached token tau < len_b,
 *   scores[b,h,tau] = sum_{hq in group(h)} sum_j q_rot[b,hq]^[dom_fc[h,j]] . k_dom[b,h,tau/64,j,tau%64,:]
 * i.e. the FC-restricted score S_t summed over the GQA group (no 1/sqrt(d)).
 */
int fasa_tip_score(const float* q_rot, const void* k_dom, const int32_t* dom_fc,
                   const int32_t* seq_lens, float* scores,
                   const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * T_t = TopK-I(S_t, N_fac) (same page, token-selection equation) per (b, KV
 * head): the min(budget, len) largest scores; equal scores keep the smaller
 * token index; -0 equals +0.  idx ascending, -1 padded; count = min(budget, len).
 */
int fasa_topk_select(const float* scores, const int32_t* seq_lens, int32_t budget,
                     int32_t* idx, int32_t* count,
                     const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * FAC (same page, §3.4 "Online Stage 2: Focused Attention Computation"): for
 * every query head, softmax(q_rot K_T^T / sqrt(d)) V_T over the rows
 * T = idx[b,h,0:count[b,h]] gathered at their original positions.
 * Indices must lie in [0, len_b).  idx rows have stride `budget`.
 */
int fasa_focused_attention(const float* q_rot, const void* k_cache, const void* v_cache,
                           const int32_t* seq_lens, const int32_t* idx, const int32_t* count,
                           int32_t budget, float* out,
                           const fasa_dims_t* dims, fasa_stream_t stream);

/* Dense full-KV decode attention (FAC with T = all tokens 0..len-1). */
int fasa_dense_attention(const float* q_rot, const void* k_cache, const void* v_cache,
                         const int32_t* seq_lens, float* out,
                         const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * One FASA decode step, fused: RoPE(q) -> TIP over k_dom -> top-k -> FAC over
 * k_cache/v_cache -> out.  idx_out / count_out may be NULL.  workspace may be
 * NULL when fasa_workspace_size reports 0.
 */
int fasa_decode_step(const void* q, const int32_t* pos,
                     const void* k_cache, const void* v_cache, const void* k_dom,
                     const int32_t* dom_fc, const int32_t* seq_lens, int32_t budget,
                     float* out, int32_t* idx_out, int32_t* count_out,
                     void* workspace, size_t workspace_bytes,
                     const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * FASA-M with split keys (same page, "Hardware-Aware Variants", FASA-M: the
 * dominant key dims C_key^dom stay on the GPU, the non-dominant ones
 * C_key^nondom and the values in CPU memory; after TIP only K^nondom_T and
 * V_T cross the link, and the keys are rebuilt with K^dom_T).
 *
 * fasa_build_knondom writes C_key^nondom: for every token tau < seq_lens[b]
 * (all tau < T_max when seq_lens is NULL), the FC pairs of
 * k_cache[b,h,tau,:] outside the head's dominant set, in FC order:
 * k_nondom[b,h,tau, 2p : 2p+2] = the p-th such pair, p < d/2 - N_tip
 * (row stride d - 2 N_tip elements, stored dtype).  k_nondom may be
 * page-locked host memory.  Every head must use exactly N_tip distinct FCs
 * (no negative entries): another table sets FASA_DEV_BAD_INPUT and leaves
 * the head's rows unwritten.  Nothing to do when N_tip = d/2.
 *
 * fasa_decode_step_split is fasa_decode_step with k_nondom in place of
 * k_cache: the FAC gathers, per selected token, its k_nondom row (d - 2 N_tip
 * elements) and its V row (d elements) -- typically from host memory -- and
 * its N_tip dominant pairs from k_dom.  Same selection; the output equals
 * the whole-key step's up to the summation order of q . k.  bf16 caches and
 * N_tip a multiple of 4 (FASA_ERR_UNSUPPORTED otherwise); the FC table as
 * for fasa_build_knondom (FASA_DEV_BAD_INPUT otherwise).
 */
int fasa_build_knondom(const void* k_cache, const int32_t* dom_fc, const int32_t* seq_lens,
                       void* k_nondom, const fasa_dims_t* dims, fasa_stream_t stream);
int fasa_decode_step_split(const void* q, const int32_t* pos,
                           const void* k_nondom, const void* v_cache, const void* k_dom,
                           const int32_t* dom_fc, const int32_t* seq_lens, int32_t budget,
                           float* out, int32_t* idx_out, int32_t* count_out,
                           void* workspace, size_t workspace_bytes,
                           const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * fasa_decode_step with the new token's cache maintenance fused in (the
 * FASA pages, "Hardware-Aware Variants": FASA-C keeps the dominant key cache
 * alongside the KV cache, so each decode step adds its own token to both).
 * For every sequence b, with t = seq_lens[b] (lengths BEFORE the step,
 * t < T_max):
 *  - k_new [B,Hkv,d] (pre-RoPE, stored dtype) is rotated by position t and
 *    written to k_cache[b,h,t,:]; v_new [B,Hkv,d] to v_cache[b,h,t,:]; the
 *    rotated key's dominant FCs to k_dom (the layout of fasa_build_kdom);
 *  - then the step runs over the t + 1 tokens 0..t with the query q at
 *    position t (the new token's own position).
 * seq_lens is read, not written: the caller advances it after the step.
 * Device-side errors (t >= T_max: nothing appended) set FASA_DEV_BAD_INPUT.
 * Same workspace and output conventions as fasa_decode_step; k_new / v_new
 * need only their element alignment.
 */
int fasa_decode_step_append(const void* q, const void* k_new, const void* v_new,
                            const int32_t* seq_lens, void* k_cache, void* v_cache, void* k_dom,
                            const int32_t* dom_fc, int32_t budget,
                            float* out, int32_t* idx_out, int32_t* count_out,
                            void* workspace, size_t workspace_bytes,
                            const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * fasa_decode_step_append_split is fasa_decode_step_append over split keys
 * (FASA-M, as fasa_decode_step_split): the rotated new key's non-dominant
 * pairs go, in FC order, to k_nondom[b,h,t,:] (row stride d - 2 N_tip, as
 * fasa_build_knondom writes it), its dominant pairs to k_dom, v_new to
 * v_cache[b,h,t,:]; then the split step runs over the t + 1 tokens.  The
 * rows written equal what fasa_build_knondom and fasa_build_kdom would
 * write from the whole rotated key.  Same restrictions and errors as
 * fasa_decode_step_split and fasa_decode_step_append.
 */
int fasa_decode_step_append_split(const void* q, const void* k_new, const void* v_new,
                                  const int32_t* seq_lens, void* k_nondom, void* v_cache, void* k_dom,
                                  const int32_t* dom_fc, int32_t budget,
                                  float* out, int32_t* idx_out, int32_t* count_out,
                                  void* workspace, size_t workspace_bytes,
                                  const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * Offline calibration of the dominant FCs (the FASA pages: "The Functional
 * Sparsity Hypothesis and the Contextual Agreement (CA) Metric", Eq. 4, and
 * the calibration procedure, Algorithm 1).
 *
 * fasa_fc_agreement: for every sequence b and KV head h, the Contextual
 * Agreement of every FC i over the cached tokens tau < len_b:
 *   alpha_i[tau] = sum over the group's query heads g of q_rot_g^[i] . k_tau^[i]
 *   full[tau]    = sum_i alpha_i[tau]        (the head's logits, group-summed
 *                                             as TIP sums them)
 *   ca[b,h,i]    = |TopK-I(full, K') & TopK-I(alpha_i, K')| / K',
 *                  K' = min(topk, len_b); 1 when len_b = 0.
 * TopK-I keeps the K' largest scores, equal scores to the smaller tau.
 *   q_rot fp32 [B,Hq,d] (rotated queries at the calibration step), k_cache as
 *   for the other entry points (16-byte aligned), ca fp32 [B,Hkv,d/2] (out).
 * dims->n_tip is not used.  The call streams K once: it writes every token's
 * full and single-FC scores into the workspace as order-preserving 32-bit
 * keys (FC-major), then each score row's TopK-I set as a token bitmask, and
 * counts the intersections from the masks (workspace:
 * B*Hkv*(d/2+1)*(T_max + T_max/32)*4 bytes).  workspace: device memory of
 * at least fasa_fc_agreement_workspace_size bytes, 16-byte aligned, owned by
 * the caller, contents not kept (FASA_ERR_WORKSPACE when missing or short).
 * Lengths out of range are clamped and set FASA_DEV_BAD_INPUT.  A calibration
 * averages ca over its samples (queries, sequences) and passes the mean to
 * fasa_select_dominant_fcs.
 */
int fasa_fc_agreement_workspace_size(const fasa_dims_t* dims, size_t* bytes);
int fasa_fc_agreement(const float* q_rot, const void* k_cache, const int32_t* seq_lens, int32_t topk,
                      float* ca, void* workspace, size_t workspace_bytes, const fasa_dims_t* dims,
                      fasa_stream_t stream);

/*
 * Compound CA of a chosen FC set (the statistic the CA page reports for the
 * dominant sets, its Table 1): Eq. 4 with alpha_i replaced by the summed
 * scores of the FCs in head h's set (dom_fc[h, :] read as above) -- the TIP
 * scores of that set:
 *   cca[b,h] = |TopK-I(full, K') & TopK-I(sum_{i in dom} alpha_i, K')| / K'.
 * Arguments as for fasa_fc_agreement; dom_fc int32 [Hkv, n_tip] (device),
 * entries >= d/2 are skipped and set FASA_DEV_BAD_INPUT; cca
 * fp32 [B, Hkv] (out).  Uses the same workspace (its size query suffices).
 */
int fasa_compound_agreement(const float* q_rot, const void* k_cache, const int32_t* dom_fc,
                            const int32_t* seq_lens, int32_t topk, float* cca, void* workspace,
                            size_t workspace_bytes, const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * Algorithm 1, last step: dom_fc[h, 0..n_tip) = the n_tip FCs of highest
 * ca_mean[h, :] (equal values: the smaller FC index first), in ascending
 * order.  ca_mean fp32 [Hkv, d/2], dom_fc int32 [Hkv, n_tip] (out), both in
 * device memory; 1 <= n_tip <= d/2.
 */
int fasa_select_dominant_fcs(const float* ca_mean, int32_t n_tip, int32_t* dom_fc,
                             const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * Size of the fixed device scratch array used by fasa_decode_step_noalloc:
 * 16 MiB, i.e. scores for B * Hkv * T_max <= 4194304 cached tokens.
 */
#define FASA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * fasa_decode_step for callers that cannot allocate device memory (the pages
 * have no counterpart: this is an interface convenience).  Same arguments as
 * fasa_decode_step without the workspace: when the step needs a score
 * workspace it uses a fixed array of FASA_NOALLOC_SCRATCH_BYTES inside the
 * library image instead (reserved on every GPU that loads the library until
 * the process exits).  Nothing is allocated or freed.
 *  - When the automatic plan (dims->reserved == 0) needs more scratch than
 *    FASA_NOALLOC_SCRATCH_BYTES, cluster sizes 2, 4, 8, 16 are tried in turn
 *    (finer token ranges need less workspace) and the first that fits runs.
 *  - Returns FASA_ERR_WORKSPACE when no plan fits the scratch (a plan that
 *    needs a workspace needs B * Hkv * T_max * 4 bytes).
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.
 *  - Every call on a device shares that device's one array: calls that may
 *    overlap on the GPU (for instance on two streams) race on it and must be
 *    serialised by the caller.  The array needs no clearing: a call writes
 *    every score it reads before reading it.
 */
int fasa_decode_step_noalloc(const void* q, const int32_t* pos,
                             const void* k_cache, const void* v_cache, const void* k_dom,
                             const int32_t* dom_fc, const int32_t* seq_lens, int32_t budget,
                             float* out, int32_t* idx_out, int32_t* count_out,
                             const fasa_dims_t* dims, fasa_stream_t stream);

/*
 * Synchronises `stream`, stores the device status word of the current device
 * in *status (FASA_DEV_* bits, 0 = clean) and clears it.  There is one word
 * per device, shared by every call on every stream of that device: a bit may
 * come from any call since the last read, and a read clears it for all of
 * them.  Callers that run steps on several streams at once read it only
 * after synchronising all of them.
 */
int fasa_device_status(fasa_stream_t stream, int32_t* status);

/*
 * Fault injection for tests (the pages have no counterpart).  Sets, for the
 * calls launched after it in this process, the bound of every device wait
 * (wait_limit_ns > 0; the default is 1 s) and:
 *  - drop_tip_tile >= 0: the fused step's TIP stage of that tile index arms
 *    its barrier but never issues the copy, so the waits on it run out;
 *  - drop_fac_refill >= 0: in the single-exchange kernel's FAC after the
 *    selection, the warp that refills attending warp 0's slots withholds
 *    its completion arrivals for that refill (0 = the first), so warp 0's
 *    wait on the slot runs out (the copies themselves are issued and land).
 * The launch then returns with FASA_DEV_TIMEOUT (with a dropped tile also
 * FASA_DEV_UNDRAINED) in the status word, no copy left in flight, and the
 * stream usable.  fasa_test_fault_injection(1000000000, -1, -1) restores
 * the defaults.  FASA_ERR_INVALID_ARG for a zero limit or an index below -1.
 */
int fasa_test_fault_injection(uint64_t wait_limit_ns, int32_t drop_tip_tile, int32_t drop_fac_refill);

/* Cluster size (CTAs per (b, KV head)) the fused kernels use on this device. */
int fasa_cluster_size(const fasa_dims_t* dims, int32_t* ctas);

/* Which fused kernel serves fasa_decode_step (and the _append and _noalloc
 * forms) for these dims on this device: FASA_KERNEL_SINGLE_EXCHANGE (bf16
 * caches, clusters of 4 or more CTAs per unit: one list exchange, a verified
 * union top-k, one combine exchange) or FASA_KERNEL_CLUSTER (every other
 * plan: the radix-select cluster kernel).  Both compute the same step; the
 * selected set and the output agree up to the documented rounding. */
enum { FASA_KERNEL_CLUSTER = 0, FASA_KERNEL_SINGLE_EXCHANGE = 1 };
int fasa_step_kernel(const fasa_dims_t* dims, int32_t* kernel);

#ifdef __cplusplus
}
#endif
#endif /* FASA_H_ */
