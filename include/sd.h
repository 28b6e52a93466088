/*
 * sd.h -- C ABI of libsd, the per-decode-step hot path of top-k sparse attention
 * (SCORE -> TOPK -> GATHER-ATT) for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (page title, section / equation):
 *   HashAttention: Semantic Sparsity for Faster Inference
 *     2.1 "inputs, outputs and the three stages" (z_i, softmax, the corrected
 *         sparse output o_hat over a selected set);
 *     2.2 "binary codes and GPU scoring" (phi(x) = ReLU(sign(F(x))), key and
 *         query encoders, SCORE = -Hamming, popcount of XOR, worked example);
 *     2.5 "why token-level sparsity runs efficiently" (page size 1: rows read
 *         in place by index; cost T = T_qmap + T_scan + T_topk + T_att);
 *     3.1 "protocol" (first 128 and last 128 tokens kept; budget counted apart).
 *   Fathom: Per-Query Read Depth for Sparse Decoding over Offloaded KV Caches
 *     paragraph "store as bit planes per channel" (4-bit codes, fp16 scale per
 *         channel per 64-token block, 4 channel-major planes, t-plane prefix is
 *         a t-bit quantiser);
 *     paragraph "per-query reverse water-filling" (gain q_j^2 sigma_j^2, each bit
 *         divides the remaining error by ~4, 0..4 bits per channel under a budget,
 *         one plan per KV head);
 *     paragraph "host planes are channel-contiguous" (one gather copies the
 *         active channels' prefixes into HBM before the scan).
 *   OasisKV: Scaling In-Decode KV Cache Beyond HBM with Lookahead Sparse Prefetching
 *     prerequisites, "sparse attention (Quest-style block summaries)" (per-block
 *         per-channel min/max, block importance, top-K blocks);
 *     method details (129 blocks of 16 tokens incl. 1 local block per KV head;
 *         UVA gather kernel from pinned CPU memory on side streams).
 *
 * Conventions (every entry point):
 *   - Ownership: the caller allocates every buffer.  libsd never allocates;
 *     scratch needs are reported by *_workspace_size().
 *   - Device pointers unless stated; 16-byte aligned.  bf16 data travel as raw
 *     bit patterns (uint16).  All layouts are row-major, last index fastest.
 *   - Asynchrony: work is enqueued on `stream` (a cudaStream_t passed as void*,
 *     NULL = legacy default stream) and the call returns without synchronising.
 *   - Errors: the return value is SD_OK or a negative SD_ERR_*; nothing is
 *     enqueued when an argument check fails.  sd_last_error() returns a
 *     thread-local message for the last failing call on this thread.
 *   - Shapes: sd_shape.d must be 128; hq % hkv == 0 and G = hq / hkv must be
 *     1, 2, 4 or 8.  n is the number of valid tokens per sequence, n_cap
 *     (>= n; 0 means n) the allocated tokens per (sequence, KV head): the
 *     stride of K, V and every per-token index buffer.
 */
#ifndef SD_H_
#define SD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SD_OK 0
#define SD_ERR_INVALID_ARG (-1) /* null pointer, bad size, bad enum, bad alignment */
#define SD_ERR_UNSUPPORTED (-2) /* a valid request outside this build (d != 128, ...) */
#define SD_ERR_CUDA (-3)        /* a CUDA call or launch failed; see sd_last_error() */
#define SD_ERR_TIMEOUT (-4)     /* a bounded wait ran out */
#define SD_ERR_WORKSPACE (-5)   /* workspace too small */

typedef struct sd_shape {
  int32_t batch; /* B: sequences in the decode batch */
  int32_t hq;    /* query heads per sequence */
  int32_t hkv;   /* KV heads per sequence */
  int32_t d;     /* head dimension (128) */
  int64_t n;     /* valid cached tokens per sequence */
  int64_t n_cap; /* allocated tokens per (sequence, KV head); 0 = n */
} sd_shape;

/* Signature encoder F (fp32, device).  hidden = 0: one projection W1 [32][d]
 * (+ b1 [32]).  hidden in {32, 64, 128}: W1 [hidden][d], b1 [hidden], ReLU,
 * W2 [32][hidden], b2 [32].  Null biases are zero. */
typedef struct sd_encoder {
  const float* W1;
  const float* b1;
  int32_t hidden;
  const float* W2;
  const float* b2;
} sd_encoder;

typedef enum {
  SD_IDX_SIG = 0,
  SD_IDX_PLANES = 1,
  SD_IDX_MINMAX = 2,
  SD_IDX_LANDMARK = 3
} sd_index_kind;
typedef enum {
  SD_PLAN_WATERFILL = 0,
  SD_PLAN_FIXED = 1,
  SD_PLAN_FULL = 2,
  SD_PLAN_TOPQ = 3,
  SD_PLAN_SPLIT = 4
} sd_plan_mode;
typedef enum { SD_SCORE_I32 = 0, SD_SCORE_F32 = 1 } sd_score_type;

/*
 * sd_build_index -- key-side index, built on the KV-write path.
 *   K: bf16 [B][hkv][n_cap][d] (tokens [0, n) are read).
 *   SD_IDX_SIG (HashAttention 2.2, eq. phi): out0 = uint32 [B][hkv][n_cap]
 *     signatures; bit o = 1 iff F_o(k) > 0.  Every dot product is the fp32 chain
 *     acc = fma(w_j, x_j, acc), j ascending from +0, then acc + bias, so the
 *     bits are reproducible on any IEEE machine.  enc is required; out1 unused.
 *   SD_IDX_PLANES (Fathom, bit planes): requires n_cap % 64 == 0.
 *     out0 = uint32 planes [B][hkv][d][4][n_cap/32] (token i = bit i%32 of word
 *     i/32; plane 0 = MSB), out1 = fp16 scales [B][hkv][d][n_cap/64] with
 *     s = f16_rn(absmax/7) (1 if that is 0) and code = clamp(rint(k/s)+8, 0, 15).
 *     A last block holding fewer than 64 tokens (n % 64 != 0) takes its scale over
 *     the tokens it holds; its bits past n are 0.  The plane scans (sd_score,
 *     sd_plan_score) read such an index at any n.  Words and scales of blocks past
 *     ceil(n/64) are not written.
 *   SD_IDX_MINMAX (OasisKV, Quest-style summaries): out0 = bf16 summaries
 *     [B][hkv][ceil(n_cap/16)][2][d]: per 16-token block the channel min row then
 *     the max row (exact keys; -0.0 orders below +0.0; the last block may be
 *     short).  out1 unused.
 *   SD_IDX_LANDMARK (the Fathom page's 8-token block landmark scan, a comparison
 *     point): out0 = bf16 landmarks [B][hkv][ceil(n_cap/8)][d]: per 8-token block
 *     the fp32 sum of its held keys in token order, divided by their count (fp32)
 *     and rounded to bf16 (nearest, ties to even).  out1 unused.
 */
int sd_build_index(int kind, const sd_shape* shape, const void* K, const sd_encoder* enc,
                   void* out0, void* out1, void* stream);

/*
 * sd_append_index -- incremental index update on the KV-write path (HashAttention
 * 2.2: signatures computed as keys are written and cached; OasisKV system design:
 * the compressed-key update).  The index in out0/out1 holds sd_build_index's result
 * for the first n_old tokens; K now holds tokens [0, n) (n = shape->n, 0 <= n_old
 * <= n, any n, typically n_old + 1 per decode step).  On return the index equals
 * sd_build_index's result for n tokens, bit for bit.  Rewritten: SD_IDX_SIG the
 * signatures of tokens [n_old, n); SD_IDX_MINMAX the 16-token blocks from
 * floor(n_old/16) on; SD_IDX_LANDMARK the 8-token blocks from floor(n_old/8) on;
 * SD_IDX_PLANES the 64-token blocks from floor(n_old/64) on (the block being filled
 * is re-quantised, since a new key can raise its scale).  Work
 * and traffic are proportional to n - n_old plus one block.  n_old == n does
 * nothing.  Arguments, layouts and errors otherwise as sd_build_index.
 */
int sd_append_index(int kind, const sd_shape* shape, int64_t n_old, const void* K,
                    const sd_encoder* enc, void* out0, void* out1, void* stream);

/*
 * sd_encode_query -- query signatures phi_q(q) (HashAttention 2.2), the
 * "query map" stage of the per-step cost.  q: bf16 [B][hq][d]; qsig: uint32
 * [B][hq].  Same fp32 chain as SD_IDX_SIG.
 */
int sd_encode_query(const sd_shape* shape, const void* q, const sd_encoder* enc,
                    uint32_t* qsig, void* stream);

/*
 * sd_plan -- per-query read plan (Fathom, reverse water-filling), one per
 * (sequence, KV head), shared by the group's query heads.
 *   q: bf16 [B][hq][d]; sigma2: fp32 [hkv][d] calibration variances;
 *   plan: uint8 [B][hkv][d], bits per channel in 0..4.
 *   SD_PLAN_WATERFILL, budget B in [0, 4d]: gain w_j = (sum_g q_gj^2) * sigma2_j
 *     in fp32 (g ascending, no fused multiply-add); the result equals giving B
 *     bits one at a time to the channel with the largest w_j * 4^-b_j among
 *     b_j < 4, lowest j on ties; sum_j plan_j = min(B, 4d).
 *   SD_PLAN_FIXED, budget r in [0, d]: the r channels with the largest sigma2_j
 *     (lowest j on ties) get 4 bits, the others 0.
 *   SD_PLAN_FULL: every channel gets 4 bits (budget ignored).
 *   SD_PLAN_TOPQ, budget r in [0, d]: the r channels with the largest query mass
 *     u_j = sum_g q_gj^2 (fp32, g ascending, no fused multiply-add; lowest j on
 *     ties) get 4 bits, the others 0: the SparQ comparison point on the Fathom
 *     page (top-r |q| channels read at full depth, r = 16 being its 68-bit
 *     setting; for G = 1 exactly the r largest |q_j|).  sigma2 is not read and may
 *     be NULL.
 *   SD_PLAN_SPLIT, budget B in [0, 4d]: the budget split across the KV heads of a
 *     sequence: its hkv * B bits go one at a time to the (head h, channel j) with
 *     the largest w_hj * 4^-b_hj among b_hj < 4 (w_hj as SD_PLAN_WATERFILL's for
 *     head h), lowest h, then lowest j, on ties; each head's sum varies, the
 *     sequence's is hkv * B.  With hkv = 1 it equals SD_PLAN_WATERFILL.  (The
 *     Fathom page keeps one budget per query and calibrates per-layer budgets;
 *     this is its marginal-gain rule over the heads of a layer.)
 * q is required by SD_PLAN_WATERFILL, SD_PLAN_TOPQ and SD_PLAN_SPLIT, sigma2 by
 * SD_PLAN_WATERFILL, SD_PLAN_FIXED and SD_PLAN_SPLIT.  Returns SD_ERR_INVALID_ARG
 * for a NULL required pointer, an unknown mode or a budget out of range, and
 * SD_ERR_UNSUPPORTED for SD_PLAN_SPLIT with hkv > 64.
 */
int sd_plan(const sd_shape* shape, const void* q, const float* sigma2, int mode, int budget,
            uint8_t* plan, void* stream);

/*
 * sd_score -- SCORE of every cached key (or block) of every (sequence, KV head).
 * Output rows are contiguous: scores [B*hkv][n] (or [B*hkv][ceil(n/16)]).
 *   SD_IDX_SIG (HashAttention 2.2): index0 = signatures, q_or_qsig = uint32
 *     qsig [B][hq]; scores int32 = -sum_{g in group} popcount(sig XOR qsig_g).
 *   SD_IDX_PLANES (Fathom): index0 = planes, index1 = scales, plan required,
 *     q_or_qsig = bf16 q [B][hq][d]; scores fp32 = sum_g sum_j q_gj *
 *     khat_ij(plan_j) with khat_t = s*(prefix_t + 2^(3-t) - 8) for t < 4 (0 for
 *     t = 0) and s*(code - 8) for t = 4, prefix_t = the code with its low 4-t
 *     bits cleared.  Only the first plan_j planes of channel j are read.
 *   SD_IDX_MINMAX (OasisKV/Quest bound): index0 = summaries, q_or_qsig = bf16
 *     q; scores fp32 [B*hkv][ceil(n/16)] = sum_g sum_j max(q_gj min_j, q_gj max_j).
 *   SD_IDX_LANDMARK: index0 = landmarks, q_or_qsig = bf16 q; scores fp32
 *     [B*hkv][ceil(n/8)] = sum_g sum_j q_gj L_j (computed as sum_j q~_j L_j with the
 *     group sum q~ in fp32).
 */
int sd_score(int kind, const sd_shape* shape, const void* index0, const void* index1,
             const void* q_or_qsig, const uint8_t* plan, void* scores, void* stream);

/*
 * sd_topk -- exact top-k per row with forced windows (HashAttention 2.1 TOPK and
 * 3.1 fixed positions; OasisKV method details: top-K blocks + 1 local block).
 *   scores: rows x n_units, SD_SCORE_I32 or SD_SCORE_F32, contiguous rows.
 *   Units are tokens (sel.block == 1) or blocks of sel.block tokens.
 *   Forced units: [0, sink) and [n_units - local, n_units).  Of the units in
 *   between, all are taken if there are at most k, else the first k in the
 *   order (score descending, unit ascending); -0.0 equals +0.0.
 *   Output: idx int32 [rows][idx_stride] holds the union in ascending order,
 *   each unit expanded to tokens [u*block, min((u+1)*block, n_tokens));
 *   count int32 [rows] = tokens written (-1 if the row holds a NaN score).
 *   Entries past count are not written.  idx_stride must be at least
 *   min(n_units, sink + local + k) * block.  Limits: 1 <= k <= 4096; n_tokens and
 *   min(n_units, sink + local + k) * block below 2^31 (SD_ERR_UNSUPPORTED).
 *   Workspace: sd_topk_workspace_size() bytes (device), contents need not be
 *   initialised; calls sharing a workspace must not overlap.
 */
typedef struct sd_select {
  int32_t k;
  int32_t sink;
  int32_t local;
  int32_t block;
} sd_select;

size_t sd_topk_workspace_size(int64_t rows, int64_t n_units, const sd_select* sel);
int sd_topk(int score_type, const void* scores, int64_t rows, int64_t n_units,
            int64_t n_tokens, const sd_select* sel, int32_t* idx, int64_t idx_stride,
            int32_t* count, void* workspace, size_t ws_bytes, void* stream);

/*
 * sd_plan_score -- sd_plan then sd_score(SD_IDX_PLANES) in one launch (Fathom's
 * per-query plan and bit-plane scan): the scan computes each row's plan from q
 * and sigma2 itself, with sd_plan's arithmetic, and writes exactly the scores the
 * two calls would.  Arguments as sd_plan (q, sigma2, mode, budget; plan may be
 * NULL, else it receives the plan) and sd_score (planes, scales, scores).
 * SD_PLAN_SPLIT couples the heads of a sequence, so it runs as sd_plan's kernel
 * and then the scan (two launches) and needs the plan buffer.
 *   Any n >= 1 (n_cap a multiple of 64).
 *   wmax: NULL, or fp32 [B*hkv][ceil(n / 32)], 4-byte aligned, receiving each
 *   32-token word's largest score over its tokens < n (NaN if one of them is NaN):
 *   the input of sd_topk_wmax.
 */
int sd_plan_score(const sd_shape* shape, const void* planes, const void* scales, const void* q,
                  const float* sigma2, int mode, int budget, uint8_t* plan, float* scores,
                  float* wmax, void* stream);

/*
 * sd_topk_wmax -- sd_topk(SD_SCORE_F32, sel.block == 1) for score rows whose
 * 32-unit maxima are known (HashAttention 2.1 TOPK over the scores of the Fathom
 * bit-plane scan): the same idx and count, drawn from the words whose maximum
 * reaches a sampled threshold instead of from every score of the row.
 *   scores fp32 [rows][n], 16-byte aligned; wmax fp32 [rows][ceil(n / 32)] with
 *   wmax[r][w] the largest of scores[r][32w .. min(32w + 31, n - 1)], NaN if one
 *   of them is NaN (as sd_plan_score writes it); any n >= 1.  Other arguments and
 *   limits as sd_topk with n_units = n_tokens = n.  Calls outside the one-CTA
 *   path (k > 1024, more than 36,864 words meeting [sink, n - local), rows of at
 *   most 8192 units, or n - sink - local <= k) run sd_topk's kernels, so the
 *   workspace is sd_topk_workspace_size(rows, n, sel) bytes.
 */
int sd_topk_wmax(const float* scores, const float* wmax, int64_t rows, int64_t n,
                 const sd_select* sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                 void* workspace, size_t ws_bytes, void* stream);

/*
 * sd_hamming_topk -- sd_score(SD_IDX_SIG) then sd_topk(SD_SCORE_I32, sel.block == 1)
 * without materialising the scores (HashAttention 2.1 SCORE -> TOPK; 2.2 SCORE =
 * -Hamming over the group's query signatures; 3.1 windows kept, budget apart): the
 * same idx and count.  Two passes over the signatures: per 8192-token range a
 * histogram of the 32G + 1 score values, then the exact k-th best value and its
 * ties (lowest index first) taken range by range in token order.
 *   sig uint32 [B][Hkv][n_cap], qsig uint32 [B][Hq] (sd_encode_query); sel with
 *   block == 1; idx int32 [B*Hkv][idx_stride], count int32 [B*Hkv], as sd_topk.
 *   workspace: device, at least sd_hamming_topk_workspace_size(shape, sel) bytes;
 *   the call resets the part it needs on the stream.
 * Errors: SD_ERR_INVALID_ARG, SD_ERR_UNSUPPORTED (k > 4096, more than 2,097,152
 * competing tokens, more than 65535 rows), SD_ERR_WORKSPACE, SD_ERR_CUDA.
 */
size_t sd_hamming_topk_workspace_size(const sd_shape* shape, const sd_select* sel);
int sd_hamming_topk(const sd_shape* shape, const uint32_t* sig, const uint32_t* qsig,
                    const sd_select* sel, int32_t* idx, int64_t idx_stride, int32_t* count,
                    void* workspace, size_t ws_bytes, void* stream);

/*
 * sd_select_attend -- sd_topk_wmax then sd_gather_attend on its result (HashAttention
 * 2.1: TOPK then GATHER-ATT; 2.5: page size 1), in one launch where one 16-CTA
 * thread-block cluster per row can run both: the same idx, count, out and lse as
 * the two calls (the selection and the attention run the same device code, with a
 * cluster barrier between them in place of a kernel boundary).
 *   scores, wmax, sel: as sd_topk_wmax with rows = B * Hkv and n = shape->n;
 *   q, K, V, scale, out, lse: as sd_gather_attend; idx [rows][idx_stride] and
 *   count [rows] receive the selection, as from sd_topk_wmax;
 *   max_count: as sd_gather_attend, with min(n, sink + local + k) <= max_count <=
 *   idx_stride.
 *   workspace: device, at least sd_select_attend_workspace_size(shape, sel,
 *   max_count) bytes (the two calls' workspaces, used where the fused launch does
 *   not apply).
 * Errors: those of the two calls.
 */
size_t sd_select_attend_workspace_size(const sd_shape* shape, const sd_select* sel,
                                       int64_t max_count);
int sd_select_attend(const sd_shape* shape, const float* scores, const float* wmax,
                     const sd_select* sel, const void* q, const void* K, const void* V,
                     float scale, int32_t* idx, int64_t idx_stride, int32_t* count,
                     int64_t max_count, float* out, float* lse, void* workspace,
                     size_t ws_bytes, void* stream);

/*
 * sd_score_topk -- sd_score(SD_IDX_PLANES) then sd_topk(SD_SCORE_F32) on those
 * scores, in one call (Fathom's bit-plane scan feeding HashAttention 2.1's TOPK):
 * writes exactly the scores, idx and count the two calls would.
 *   Arguments as sd_score with kind SD_IDX_PLANES (planes, scales, q, plan;
 *   scores fp32 [B*hkv][n]) and as sd_topk with rows = batch * hkv and
 *   n_units = n_tokens = n; sel.block must be 1.
 *   Rows of at least 65536 competing tokens (n - sink - local) with n_cap a
 *   multiple of 512 and 16-byte aligned planes and scales take a fused path: a
 *   sample of each row (512 runs of 32 tokens, scored with the plan) sets a
 *   threshold below the row's k-th score with high probability, the scan marks
 *   every competing token that reaches it (one bit per token), and the top k are
 *   drawn from the marked tokens instead of from a second pass over the scores;
 *   a row with fewer than k marks, more than the selection can gather, or a NaN
 *   is selected from its full score row.  Other calls run the scan, then
 *   sd_topk's kernels.
 *   Workspace: sd_score_topk_workspace_size() bytes of device memory, 256-byte
 *   aligned; contents need not be initialised; calls sharing a workspace must
 *   not overlap.
 */
size_t sd_score_topk_workspace_size(const sd_shape* shape, const sd_select* sel);
int sd_score_topk(const sd_shape* shape, const void* planes, const void* scales, const void* q,
                  const uint8_t* plan, const sd_select* sel, float* scores, int32_t* idx,
                  int64_t idx_stride, int32_t* count, void* workspace, size_t ws_bytes,
                  void* stream);

/*
 * sd_gather_attend -- GATHER-ATT (HashAttention 2.1, corrected o_hat; 2.5 page
 * size 1): for query head g of sequence b, KV head h = g / G, over the rows
 * I = idx[b*hkv + h][0..count): z_i = scale * <q_g, k_i>,
 * out = sum_i e^{z_i - m} v_i / sum_i e^{z_i - m}, lse = m + log(sum e^{z_i - m}).
 *   q bf16 [B][hq][d]; K, V bf16 [B][hkv][n_cap][d]; idx int32 [B*hkv][idx_stride]
 *   (token indices < n, any order); count int32 [B*hkv] (<= max_count);
 *   out fp32 [B][hq][d]; lse fp32 [B][hq] or NULL.  An empty set gives out = 0,
 *   lse = -inf.  The set is split across CTAs (or warps) and merged by an
 *   online-softmax combine: a few rows go to one thread-block cluster per row;
 *   many long rows (at least 4 groups of 16 selected tokens per warp of a full
 *   grid, with q 16-byte aligned) go to a persistent kernel whose warps each take
 *   an equal range of 16-token groups and run QK^T and PV on the tensor cores,
 *   their partials combined through the workspace.  Workspace:
 *   sd_gather_attend_workspace_size() bytes (device).
 */
size_t sd_gather_attend_workspace_size(const sd_shape* shape, int64_t max_count);
int sd_gather_attend(const sd_shape* shape, const void* q, const void* K, const void* V,
                     const int32_t* idx, int64_t idx_stride, const int32_t* count,
                     int64_t max_count, float scale, float* out, float* lse, void* workspace,
                     size_t ws_bytes, void* stream);

/*
 * sd_gather_attend_noalloc -- sd_gather_attend for callers that cannot allocate
 * device memory or hand the library a workspace: engines whose host framework
 * owns every device allocation (a pool or custom allocator the library must not
 * bypass), real-time loops that must not take allocator locks or let cudaMalloc
 * synchronise the device, and code that runs where cudaMalloc may not be called.
 * (The pages have no counterpart: this is a property of the library, not of the
 * method.)
 *   Same arguments, layouts and results as sd_gather_attend, without the
 *   workspace: when the split-n or the many-row kernel runs, its ticket and
 *   partials live in a 4 MiB file-scope device array that every GPU loading libsd
 *   holds until the process exits.  The limit is applied to every call, whichever kernel then runs:
 *   requests whose partials would need more (sd_gather_attend_workspace_size()
 *   > 4 MiB) are rejected with SD_ERR_UNSUPPORTED before anything is enqueued,
 *   so a call that succeeds on one GPU succeeds on every GPU.  Allocates nothing.
 *   The first call on each device looks up that device's copy of the array
 *   (cudaGetSymbolAddress, with the device current) and keeps the address for
 *   the process; make that first call before any stream capture.  A device
 *   reset (cudaDeviceReset) invalidates the kept address: do not call this entry
 *   point on a device after resetting it.  When the 16-CTA cluster kernel runs,
 *   the array is not used.  When another kernel runs, all calls
 *   on a device share the array and it keeps the last call's contents: each such
 *   call first clears the per-row counters that must start at zero (on the
 *   caller's stream; partials are written before they are read), and calls that
 *   overlap on the GPU race on it.
 */
int sd_gather_attend_noalloc(const sd_shape* shape, const void* q, const void* K, const void* V,
                             const int32_t* idx, int64_t idx_stride, const int32_t* count,
                             int64_t max_count, float scale, float* out, float* lse,
                             void* stream);

/*
 * sd_offload_gather -- copy each (sequence, KV head, channel j)'s planned
 * prefix (the first plan_j planes, contiguous in the channel-major layout)
 * and channel j's scales from pinned host memory into HBM, with device loads
 * over the host link (Fathom, host planes; OasisKV, UVA gather on a side stream).
 *   host_planes / host_scales: pinned host memory (cudaHostAlloc or registered)
 *   in the SD_IDX_PLANES layout; plan: device uint8 [B][hkv][d];
 *   dev_planes / dev_scales: device buffers in the same layout.  Channels with
 *   plan_j = 0 and planes past the prefix are not written.  Typically enqueued
 *   on a side stream; the caller orders the scan after it with an event.
 */
int sd_offload_gather(const sd_shape* shape, const uint32_t* host_planes,
                      const uint16_t* host_scales, const uint8_t* plan, uint32_t* dev_planes,
                      uint16_t* dev_scales, void* stream);

/*
 * Resident set of the delta selection (OasisKV method details: the GPU keeps a
 * fixed pool of blocks per KV head -- 129 blocks of 16 tokens there -- and a head-
 * level map from logical blocks to pool pages).  Device arrays owned by the
 * caller, rows = B * hkv; every entry -1 for an empty set (fill the bytes with 0xFF):
 *   slot_unit int32 [rows][n_slots]  unit held by each slot, -1 empty;
 *   slot_last int32 [rows][n_slots]  step at which that unit was last selected;
 *   unit_slot int32 [rows][n_units]  slot holding each unit, -1 not resident.
 */
typedef struct sd_resident {
  int32_t n_slots;
  int32_t* slot_unit;
  int32_t* slot_last;
  int32_t* unit_slot;
} sd_resident;

/*
 * sd_delta_select -- the KV-selection step (OasisKV method details): intersect the
 * predicted units with the resident set and plan at most admit_cap admissions per
 * (sequence, KV head), each evicting the least-recently-selected slot outside the
 * prediction.
 *   shape: n tokens; units are blocks of sel->block tokens, n_units =
 *   ceil(n / block).  scores: fp32 [rows][n_units] and idx/count: the sd_topk
 *   output over those scores (tokens of each unit expanded, ascending; a unit is
 *   predicted when its first token is listed).  A row with count < 0 is left
 *   alone (plan_count = pool_count = -1).
 *   Hits (predicted and resident) stay where they are; their slot_last becomes
 *   step.  Misses are admitted in order: forced units (sel's sink and local
 *   windows) unit ascending, then score descending, unit ascending (-0.0 equals
 *   +0.0).  Targets: the slots not holding a predicted unit, by slot_last
 *   ascending (empty slots first), slot ascending.  a = min(admit_cap, misses,
 *   targets) pairs are made; slot_last of each taken slot becomes step.
 *   Outputs: plan_slot / plan_unit / plan_evict int32 [rows][admit_cap] (entries
 *   past plan_count not written; plan_evict = the unit evicted or -1) and
 *   plan_count [rows]; pool_idx int32 [rows][pool_stride]: the pool rows
 *   slot*block + t of every predicted unit resident after the step, in unit order
 *   (t < the unit's token count), pool_count [rows] (the input of sd_gather_attend
 *   over the pool).
 *   Limits: 1 <= block <= 4096; min(n_units, sink + local + k) <= 8192 units;
 *   1 <= n_slots <= 4096; 0 <= admit_cap <= 8192; 0 <= step < 2^31 - 1;
 *   idx_stride and pool_stride at least min(n_units, sink + local + k) * block.
 *   Steps of one resident set must not overlap.  The state is read as it stands:
 *   a map entry that disagrees with its slot counts as not resident, so no state
 *   content can make the kernel access memory outside the arrays.
 *   Errors (nothing is launched): SD_ERR_INVALID_ARG for a NULL required pointer
 *   (plan arrays are required when admit_cap > 0), a bad sel, admit_cap, step or
 *   stride; SD_ERR_UNSUPPORTED for n_slots or the predicted-unit bound outside
 *   the limits; SD_ERR_CUDA if the launch fails.  All arrays are device memory
 *   owned by the caller.
 */
int sd_delta_select(const sd_shape* shape, const sd_select* sel, const float* scores,
                    const int32_t* idx, int64_t idx_stride, const int32_t* count,
                    int32_t admit_cap, int32_t step, const sd_resident* res,
                    int32_t* plan_slot, int32_t* plan_unit, int32_t* plan_evict,
                    int32_t* plan_count, int32_t* pool_idx, int64_t pool_stride,
                    int32_t* pool_count, void* stream);

/*
 * sd_resident_gather -- the KV-transfer step (OasisKV: a UVA gather kernel writes
 * the planned blocks from pinned CPU memory into the GPU's resident pages): for
 * each plan entry i < plan_count of each row, the unit's tokens [u*block,
 * min((u+1)*block, n)) of K and V are copied to pool rows slot*block..; rows of a
 * short last unit past n are written as zeros.
 *   K, V: bf16 [B][hkv][n_cap][d], device memory or pinned host memory (cudaHostAlloc
 *   or registered); K_pool, V_pool: device bf16 [B][hkv][n_slots * block][d].  All
 *   16-byte aligned.  Entries with a slot or unit out of range are skipped.
 *   Errors: SD_ERR_INVALID_ARG for a NULL or misaligned pointer, a block outside
 *   [1, 4096], admit_cap outside [0, 8192] or K/V that are neither device nor
 *   pinned host memory; SD_ERR_UNSUPPORTED for n_slots outside [1, 4096].
 */
int sd_resident_gather(const sd_shape* shape, int32_t block, const void* K, const void* V,
                       const int32_t* plan_slot, const int32_t* plan_unit,
                       const int32_t* plan_count, int32_t admit_cap, int32_t n_slots,
                       void* K_pool, void* V_pool, void* stream);

/*
 * One sequence split by tokens across devices (HashAttention 2.5: contexts beyond
 * one device).  Shard s holds tokens [a_s, a_s + n_s) of the sequence with its own
 * index, K and V (cut at whole 64-token blocks, so its bit-plane scores are the
 * unsharded ones); the forced windows [0, lead) and [tail, n) stay with the shards
 * holding them, as (sink_s, local_s) in the shard's own indices.  A step: each shard
 * runs its plan, scan and sd_topk with (k, sink_s, local_s); sd_shard_candidates;
 * an all-gather of the candidates; sd_topk_merge (every shard the same result);
 * sd_shard_select; sd_gather_attend on the shard's set; an all-gather of (out, lse);
 * sd_attend_combine.  The result equals the unsharded step's selection exactly and
 * its attention within rounding.
 *
 * sd_shard_candidates -- the shard's competing tokens of its own top-k: the entries
 *   of idx [rows][idx_stride] (ascending, count [rows]) in [sink_s, n_s - local_s),
 *   in their order, with scores [rows][n_s] (fp32) and global index offset + t:
 *   cand_score fp32 [rows][k], cand_idx int32 [rows][k], cand_count [rows] (-1 for a
 *   row whose count is -1).  Entries past cand_count are not written.
 */
int sd_shard_candidates(const float* scores, int64_t rows, int64_t n_s, const int32_t* idx,
                        int64_t idx_stride, const int32_t* count, int32_t sink_s, int32_t local_s,
                        int64_t offset, int32_t k, float* cand_score, int32_t* cand_idx,
                        int32_t* cand_count, void* stream);

/*
 * sd_topk_merge -- the sequence's top-k from every shard's candidates:
 *   cand_score fp32 [shards][rows][k], cand_idx int32 [shards][rows][k], cand_count
 *   int32 [shards][rows] (as sd_shard_candidates writes them, gathered).  Of their
 *   union, the first k in the order (score descending, index ascending; -0.0 equals
 *   +0.0) are written ascending to idx [rows][idx_stride >= k]; count [rows] = their
 *   number, -1 if any shard's count is -1.  shards * k <= 8192.
 */
int sd_topk_merge(int64_t rows, int32_t shards, int32_t k, const float* cand_score,
                  const int32_t* cand_idx, const int32_t* cand_count, int32_t* idx,
                  int64_t idx_stride, int32_t* count, void* stream);

/*
 * sd_shard_select -- the shard's attention set in its own indices, ascending:
 *   [0, sink_s), the merged tokens (sel_idx [rows][sel_stride], sel_count [rows],
 *   global, ascending, at most k) that lie in [offset, offset + n_s) shifted by
 *   -offset, and [n_s - local_s, n_s); idx [rows][idx_stride >= sink_s + local_s +
 *   k], count [rows] (-1 where sel_count is -1).  The input of sd_gather_attend over
 *   the shard's K and V.
 */
int sd_shard_select(int64_t rows, const int32_t* sel_idx, int64_t sel_stride,
                    const int32_t* sel_count, int64_t offset, int64_t n_s, int32_t sink_s,
                    int32_t local_s, int32_t k, int32_t* idx, int64_t idx_stride, int32_t* count,
                    void* stream);

/*
 * sd_attend_combine -- the split-softmax combine of the shards' attention over
 *   disjoint token sets: outs fp32 [shards][batch][hq][128] and lses fp32
 *   [shards][batch][hq] as sd_gather_attend writes them; with L = log sum_s
 *   exp(lse_s), out = sum_s exp(lse_s - L) out_s and lse = L (lse may be NULL).
 *   Shards with an empty set (lse = -inf) weigh 0; all empty give out = 0, lse =
 *   -inf.
 */
int sd_attend_combine(int32_t shards, int64_t batch, int32_t hq, const float* outs,
                      const float* lses, float* out, float* lse, void* stream);

/*
 * sd_device_status -- device-side errors of the work already enqueued on
 * `stream`: waits for the stream, then reads and clears this GPU's libsd error
 * word.  Every wait inside libsd's kernels is bounded; one that runs out (a
 * bulk copy that never lands) makes the kernel stop its work early and set the
 * word instead of hanging.  Returns SD_OK, SD_ERR_TIMEOUT when a kernel gave up
 * since the last check (its outputs are incomplete; message in sd_last_error()),
 * or SD_ERR_CUDA when the stream reports an error.  Synchronises `stream`: call
 * it between steps, not inside a captured graph.
 */
int sd_device_status(void* stream);

/*
 * sd_set_fallback_paths -- testing switch (process-wide, off by default): while
 * on, sd_gather_attend (and its no-allocation variant), the top-k entry points
 * and the bit-plane scans take the kernels they use on GPUs where their
 * thread-block clusters cannot be co-resident or bulk copies do not apply: the
 * split-n gather-attend with workspace partials, the sampled-threshold
 * sample/filter/finish top-k, the one-CTA word-maxima top-k, sd_select_attend
 * as its two calls, and the cp.async bit-plane scan.  Results are the same.
 * Returns the previous setting.
 */
int sd_set_fallback_paths(int on);

/*
 * sd_debug_set_device_error -- testing: sets this GPU's libsd error word as a
 * kernel whose bounded wait ran out would (ordered on `stream`, then waits for
 * it), so that sd_device_status's report can be tested without making a wait
 * run out.
 */
int sd_debug_set_device_error(void* stream);

/*
 * sd_copy -- copy `bytes` bytes from src to dst with a kernel on `stream`, where
 * each pointer is device memory or pinned host memory that the device reaches
 * at the same address (unified addressing: cudaHostAlloc / pin_memory buffers).
 * For a decode step's small inputs and results: inside a CUDA graph a copy
 * kernel over the pinned memory's mapping finishes sooner than a copy-engine
 * transfer.  Both pointers 16-byte aligned, bytes a multiple of 16
 * (SD_ERR_INVALID_ARG otherwise); the ranges must not overlap; bytes = 0 does
 * nothing.
 */
int sd_copy(void* dst, const void* src, size_t bytes, void* stream);

/*
 * sd_event_wait -- host-side bounded wait on a cudaEvent_t (passed as void*):
 * polls until the event completes or timeout_us microseconds pass
 * (SD_ERR_TIMEOUT).  Lets a caller bound its wait for an offload copy.
 */
int sd_event_wait(void* event, int64_t timeout_us);

/* Thread-local message of the last failing call on this thread ("" if none). */
const char* sd_last_error(void);

/* ABI version (major * 100 + minor): 101 adds sd_append_index, SD_PLAN_TOPQ,
 * SD_IDX_LANDMARK, sd_delta_select and sd_resident_gather to 100; 102 adds
 * sd_device_status, sd_set_fallback_paths and sd_debug_set_device_error; 103 adds
 * SD_PLAN_SPLIT, sd_shard_candidates, sd_topk_merge, sd_shard_select and
 * sd_attend_combine; 104 adds sd_copy. */
int sd_version(void);

/*
 * sd_launch_count -- number of kernels this library has launched in this
 * process (all devices and threads; a graph replay launches nothing through
 * the library and is not counted).  Read it before and after a call to count
 * that call's launches.
 */
int64_t sd_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SD_H_ */
