/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * What the library computes
 * -------------------------
 * Scaled-dot-product attention, exactly (up to floating-point rounding):
 *
 *     S = scale * Q K^T  (+ causal mask: key j hidden from query i when j > i)
 *     O = softmax_rows(S) V,        LSE_i = log( sum_j exp(S_ij) )
 *
 * "Attention at Scale -- From FlashAttention to FlashAttention-4", section
 * "The Problem", gives the definition (score matrix, softmax, product with V);
 * the section "The Evolution" gives the tiled computation with a running
 * row max and sum ("online softmax") that keeps the N x N matrix out of HBM.
 * "FlashAttention 3 and 4: When the Bottleneck Moves", section 3.2, and the
 * abstract of "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design
 * for Asymmetric Hardware Scaling" give the forward's exponential split
 * (hardware unit plus polynomial) and conditional rescaling; the same paper's
 * Figure 2 and Table 3 give the backward's five matrix products, and its
 * abstract and Figures 7-8 the atomic and deterministic dQ accumulation.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are dense, contiguous, row-major [B, H, N, d] arrays of bfloat16
 *   in device memory (Q, K: d = d_qk; V, O, dO: d = d_v); LSE is FP32
 *   [B, H, N].  N is the same for queries and keys.
 * - Every device pointer must be 16-byte aligned.
 * - Supported head dims (d_qk, d_v): (64, 64), (128, 128), (192, 128) for the
 *   forward and the backward; the masked, FP8 and split-KV entry points list
 *   their own.
 * - B, H, N >= 1; B * H < 2^31; N < 2^24.
 * - The caller owns every buffer, including the backward workspace.  The
 *   library allocates no device memory; it keeps one device status word per
 *   GPU.
 * - Work is enqueued on ``stream`` (a cudaStream_t; NULL = legacy default
 *   stream) and the call returns without synchronising.  Argument errors are
 *   returned synchronously and nothing is launched.  Launch failures return
 *   ATTN_ERR_CUDA.  Errors found by the kernels (a wait that ran past its time
 *   limit) are recorded in the device status word; read them with
 *   attn_get_device_status.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, size out of range, non-finite scale, bad flag */
  ATTN_ERR_UNSUPPORTED = 2, /* head-dim pair not built */
  ATTN_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  ATTN_ERR_WORKSPACE = 4,   /* backward workspace missing or smaller than attn_bwd_workspace_bytes */
  ATTN_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed */
  ATTN_ERR_TIMEOUT = 6,     /* device: a pipeline wait exceeded its time limit; outputs are invalid */
  ATTN_ERR_BOUNDS = 7       /* device: an internal consistency check failed; outputs are invalid */
} attn_status_t;

/*
 * Forward pass.
 *   q [B,H,N,d_qk], k [B,H,N,d_qk], v [B,H,N,d_v]   bf16, read only
 *   o [B,H,N,d_v]  bf16, written (softmax(S) V, normalised)
 *   lse [B,H,N]    fp32, written: natural-log log-sum-exp of the scaled,
 *                  unmasked scores of each query row (what the backward needs)
 *   causal         0 or 1 (top-left aligned: query i sees keys 0..i)
 *   scale          finite and > 0; usually 1/sqrt(d_qk)
 * Returns ATTN_OK or an argument / launch error (see the enum).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d_qk,
             int d_v, int causal, float scale, cudaStream_t stream);

/*
 * Forward with grouped-query attention (the K/V-head sharing that "Attention
 * at Scale -- From FlashAttention to FlashAttention-4", section
 * "Sequence-Aware Split Heuristic", names as GQA/MQA): H query heads share
 * H_kv K/V heads, query head h reading K/V head h / (H / H_kv).
 *   q, o [B,H,N,d], lse [B,H,N]; k, v [B,H_kv,N,d]; H % H_kv == 0 (H_kv = H
 *   is attn_fwd, H_kv = 1 multi-query attention).  Other arguments as attn_fwd.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                 int d_qk, int d_v, int causal, float scale, cudaStream_t stream);

/*
 * Bytes of device workspace attn_bwd needs for these sizes (0 for sizes the
 * backward does not accept).  The workspace holds, per (b, h): the FP32 row
 * terms D_i = dO_i . O_i and LSE_i * log2(e) (padded to a multiple of 128
 * rows), the FP32 dQ accumulator, and (deterministic mode) one int32 ticket per
 * 128-row query tile.  With atomic dQ at d_qk = d_v = 64 or 128 it also holds
 * the region where the persistent backward kernel leaves the pieces of the
 * units it cuts in its last round: FP32 dV and dK partials of 128 rows per
 * piece, for min(160, B*H*ceil(N/128) - 1) pieces.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d_qk, int d_v, int deterministic);

/*
 * Backward pass: gradients of the forward with respect to q, k, v given dO.
 *   q, k, v, o, dO  bf16 [B,H,N,d] as in attn_fwd (o is the forward's output)
 *   lse             fp32 [B,H,N] from attn_fwd with the same arguments
 *   dq, dk, dv      bf16 [B,H,N,d], overwritten (not accumulated); dq and dk
 *                   are d_qk wide, dv is d_v wide
 *   (d_qk, d_v) = (192, 128) runs a kernel of its own: dV and dK (128 + 192
 *   columns) stay in tensor memory while S^T and dP^T take turns in one
 *   128-column region (the five products of "FlashAttention-4: Algorithm
 *   and Kernel Pipelining Co-Design for Asymmetric Hardware Scaling",
 *   Figure 2, unchanged).
 *   deterministic   0: dQ partial sums are added in whatever order the tiles
 *                      finish (results may differ in the last bits run to run);
 *                   1: the additions into each dQ tile happen in a fixed
 *                      order, so repeated calls give bit-identical dq, dk, dv.
 *   workspace       device memory of at least attn_bwd_workspace_bytes bytes,
 *                   16-byte aligned, owned by the caller, contents ignored on
 *                   entry and clobbered.
 * Returns ATTN_OK or an argument / launch error.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int N, int d_qk, int d_v, int causal, float scale,
             int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Masked attention ("Attention at Scale -- From FlashAttention to
 * FlashAttention-4", FlexAttention section: variants such as sliding windows
 * as a boolean mask over (query, key) pairs, plus a precomputed block map
 * whose empty blocks the kernel skips).  Query i sees key j when
 *     i - window_left <= j <= i + window_right     (-1: unbounded on that side)
 * and block_mask[(i / 128) * T + j / 128] != 0, T = ceil(N / 128).
 *   window_left, window_right   >= -1 (left = -1, right = 0 is the causal mask)
 *   block_mask   device uint8 [T, T], 16-byte aligned, shared by every (b, h),
 *                or NULL (all tiles allowed)
 * Only the tile pairs holding a visible pair are computed; pairs are masked
 * individually inside tiles the window does not cover whole.  A query row
 * with no visible key gets O = 0 and LSE = -inf (and zero dQ).  Other
 * arguments, layouts and the backward workspace are those of attn_fwd /
 * attn_bwd; d_qk = d_v = 64 or 128.  The forward runs one 128-row query tile
 * per CTA; the backward uses the one-CTA kernel (attn_set_bwd_pair does not
 * apply).  Returns ATTN_OK or an argument / launch error.
 */
int attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d_qk,
                    int d_v, int window_left, int window_right, const unsigned char* block_mask, float scale,
                    cudaStream_t stream);

int attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int H, int N, int d_qk, int d_v, int window_left,
                    int window_right, const unsigned char* block_mask, float scale, int deterministic,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Split-KV forward ("Attention at Scale -- From FlashAttention to
 * FlashAttention-4": the FlashInfer section's associative merge of attention
 * over disjoint key sets, and the "Sequence-Aware Split Heuristic" section's
 * split of the key sequence over thread blocks when B * H is too small to
 * fill the GPU, e.g. in decode).  Non-causal attention of N_q queries over
 * N_k keys:
 *   q [B,H,N_q,d_qk], k [B,H,N_k,d_qk], v [B,H,N_k,d_v]   bf16, read only
 *   o [B,H,N_q,d_v] bf16 and lse [B,H,N_q] fp32, written as by attn_fwd
 *   n_splits        requested number of key ranges (>= 1).  The keys are cut
 *                   into ceil(N_k/128) tiles of 128 and the tiles into ranges
 *                   of ceil(tiles / min(n_splits, tiles)) tiles, the last one
 *                   ragged, so that no range is empty; the number of ranges
 *                   used can be below n_splits.
 *   workspace       device memory of at least attn_fwd_splitkv_workspace_bytes
 *                   bytes, 16-byte aligned, caller-owned, clobbered: the
 *                   ranges' FP32 outputs and LSEs.
 * Two kernels run on ``stream``: the forward kernel computes every (b, h,
 * query block, key range) part, then the merge (attn_merge) combines the
 * parts of each row; the merge is launched as a programmatic dependent launch
 * (it starts while the forward drains and waits for its results inside), or
 * as an ordinary launch where the stream does not allow that.  The head dims are attn_fwd's.  Returns ATTN_OK or an
 * argument / launch error.
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N_q,
                     int N_k, int d_qk, int d_v, float scale, int n_splits, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/*
 * Split-KV forward with grouped-query attention (decode with few K/V heads,
 * the case the sequence-aware split section describes): q, o [B,H,N_q,d],
 * lse [B,H,N_q], k, v [B,H_kv,N_k,d], H % H_kv == 0.  The H / H_kv query heads
 * of one K/V head are contiguous rows of q, so this is exactly
 * attn_fwd_splitkv over B * H_kv heads of (H / H_kv) * N_q query rows (each
 * K/V tile is read once per group, not once per query head): size the
 * workspace with attn_fwd_splitkv_workspace_bytes(B, H_kv, (H / H_kv) * N_q,
 * N_k, d_v, n_splits) and choose n_splits with attn_splitkv_heuristic(B,
 * H_kv, (H / H_kv) * N_q, N_k, d_qk, n_sms).
 */
int attn_fwd_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv,
                         int N_q, int N_k, int d_qk, int d_v, float scale, int n_splits, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes attn_fwd_splitkv needs for these sizes and this requested
 * n_splits (0 for arguments it rejects): 4 * R * (d_v + 1) rounded up, with
 * R = ranges used * B * H * N_q.
 */
size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N_q, int N_k, int d_v, int n_splits);

/*
 * Number of key ranges for attn_fwd_splitkv on a GPU with n_sms
 * multiprocessors, following the sequence-aware split heuristic.  The
 * forward runs (b, h, query block) units: blocks of one 128-row query tile
 * when N_q <= 128 and d_qk <= 128 (two CTAs per multiprocessor), else of two
 * tiles (one CTA per multiprocessor); S = n_sms times the CTAs per
 * multiprocessor.  With U units, the answer is the largest power of two n
 * with n * U <= S (1 when 2U > S), so that every part runs in one wave,
 * capped so each range is at least two key tiles long.  Pure host
 * computation.  Returns 0 for invalid arguments (including a d_qk attn_fwd
 * does not support).
 */
int attn_splitkv_heuristic(int B, int H, int N_q, int N_k, int d_qk, int n_sms);

/*
 * Merge of attention partials over disjoint key sets (the associative merge
 * operator of the FlashInfer section cited above): for every row r,
 *   LSE_r = log sum_s exp(lse_parts[s,r]),
 *   O_r   = sum_s exp(lse_parts[s,r] - LSE_r) o_parts[s,r,:].
 *   o_parts [n_parts, BH*N, d_v] fp32 and lse_parts [n_parts, BH*N] fp32
 *     (natural log; a part with LSE = -inf holds no key and drops out)
 *   o [BH*N, d_v] bf16 and lse [BH*N] fp32, written (a row whose parts are all
 *     empty gets O = 0, LSE = -inf)
 *   n_parts >= 1, BH * N < 2^33, d_v 64 or 128; device pointers 16-byte
 *   aligned.  Returns ATTN_OK or an argument / launch error.
 */
int attn_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse, int BH, int N,
               int d_v, cudaStream_t stream);

/*
 * FP8 (e4m3) forward ("FlashAttention 3 and 4: When the Bottleneck Moves",
 * section 2.2: per-block scales, and a fixed random rotation R of Q and K
 * before quantising, which leaves every score unchanged since
 * (QR)(KR)^T = Q K^T).  Two calls: attn_fp8_quantize turns bf16 Q, K, V
 * into e4m3 codes with scales, attn_fwd_fp8 runs the forward on them.
 * d_qk = d_v = 128 only.
 *
 * Bytes of device workspace attn_fp8_quantize needs (0 for invalid sizes).
 */
size_t attn_fp8_quantize_workspace_bytes(int B, int H);

/*
 * Quantiser.  R = D H / sqrt(d): H the d x d Sylvester-Hadamard matrix
 * (H_ij = (-1)^popcount(i & j)), D = diag(signs).
 *   q, k, v        bf16 [B,H,N,d] device, read only
 *   signs          HOST array of d entries, each +1 or -1 (read during the
 *                  call); the same signs must be used for every call whose
 *                  codes meet in one forward
 *   q8, k8         uint8 [B,H,N,d] device, written: e4m3 codes of
 *                  (x sqrt(d) R) / s for the rows of Q and K (sqrt(d) R = D H
 *                  is exact in binary arithmetic)
 *   v8             uint8 [B,H,N,d] device, written: e4m3 codes of v / s
 *   sq, sk         fp32 [B,H,ceil(N/128)] device, written: one scale s per
 *                  128-row tile of Q and of K
 *   sv             fp32 [B,H] device, written: one scale per (b, h) of V
 *   workspace      device, >= attn_fp8_quantize_workspace_bytes, clobbered
 * Scales are powers of two, the smallest with max|x| <= 448 s over the block
 * (1 for an all-zero block); codes round to nearest even and saturate at
 * +-448.  Three kernels (a memset of the workspace, the per-head max of |V|,
 * the quantiser) run on ``stream``.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG
 * (null pointer, bad sign, sizes), ATTN_ERR_UNSUPPORTED (d != 128),
 * ATTN_ERR_MISALIGNED, ATTN_ERR_WORKSPACE or ATTN_ERR_CUDA.
 */
int attn_fp8_quantize(const void* q, const void* k, const void* v, const signed char* signs, void* q8, void* k8,
                      void* v8, float* sq, float* sk, float* sv, int B, int H, int N, int d, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/*
 * FP8 forward from attn_fp8_quantize's outputs: O = softmax(scale Q K^T
 * (+ causal mask)) V and LSE as attn_fwd, with the products on e4m3 operands
 * (FP32 accumulation) and P rounded to e4m3.  The running row max m moves
 * only when it rises by more than tau = 4 (log2 units; the decision is taken
 * per group of 32 query rows), so P <= 2^4 against the stale max and
 * P' = 2^(x - m + 4) <= 2^8 is stored as e4m3(P'); the row sum takes P'
 * before rounding, and O = s_v (sum P'_e4m3 v8) / sum P'.  (The environment
 * variable ATTN_FP8_TAU = 0..8, read at first use, changes tau.)
 *   o bf16 [B,H,N,d], lse fp32 [B,H,N] written; other arguments as attn_fwd.
 * Returns ATTN_OK or an argument / launch error.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk, const float* sv,
                 void* o, float* lse, int B, int H, int N, int d, int causal, float scale, cudaStream_t stream);

/*
 * Backward with grouped-query attention: gradients of attn_fwd_gqa.
 *   q, o, dO, dq [B,H,N,d], lse [B,H,N]; k, v, dk, dv [B,H_kv,N,d];
 *   H % H_kv == 0.  dk and dv of a K/V head sum the contributions of its
 *   H / H_kv query heads.  Workspace: attn_bwd_workspace_bytes(B, H, N, ...)
 *   (per query head).  Other arguments as attn_bwd (the CTA-pair mode does
 *   not apply).
 */
int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d_qk, int d_v, int causal,
                 float scale, int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronises ``stream``, then returns and clears the device status word of
 * the current device: ATTN_OK, or the first error a kernel recorded since the
 * last call (ATTN_ERR_TIMEOUT, ATTN_ERR_BOUNDS).  If the stream itself
 * reports a CUDA error, returns ATTN_ERR_CUDA.  ``where`` (may be NULL)
 * receives the kernel's code for the wait or check that failed.
 */
int attn_get_device_status(cudaStream_t stream, int* where);

/* Static, human-readable name of a status code. */
const char* attn_status_string(int status);

/*
 * Accuracy probe of the exponential paths the forward uses.  Writes
 * out[i] = 2^x[i] computed by ``method``: 0 = the hardware MUFU ex2.approx,
 * 3 / 4 / 5 = the polynomial emulation of that degree (2^floor(x) * p(frac)).
 * x and out are device FP32 arrays of n elements.  The cubic is the one the
 * forward kernel uses.  "FlashAttention-4 ...", Table 2, reports the same
 * measurement.
 */
int attn_exp2_probe(const float* x, float* out, int n, int method, cudaStream_t stream);

/*
 * Throughput probe: one launch over ``blocks`` blocks of 256 threads, each
 * thread evaluating ``iters`` chained exponentials by ``method`` (as above).
 * ``sink`` (device, >= blocks*256 floats) receives the results so the work is
 * kept.  Time it with events on ``stream``.
 */
int attn_exp2_throughput(float* sink, int blocks, int iters, int method, cudaStream_t stream);

/*
 * Forward-pass rescale counter: when ``counter`` is a non-NULL device
 * pointer, later attn_fwd calls on this device add to it the number of
 * (row, key-tile) steps at which the running max rose by more than the
 * threshold and the row was rescaled (first tiles not counted).  NULL turns
 * counting off.  Returns ATTN_OK.
 */
int attn_set_rescale_counter(unsigned long long* counter);

/*
 * Threshold, in log2 units, for the conditional rescale of the running
 * softmax state (default 8.0, i.e. a factor of 256; 0 rescales on every rise
 * of the max).  Must be finite and in [0, 16].  Applies to later attn_fwd calls.
 */
int attn_set_rescale_threshold(float tau);

/*
 * Exponential path of the bf16 forward ("FlashAttention-4: Algorithm and
 * Kernel Pipelining Co-Design for Asymmetric Hardware Scaling", abstract and
 * Table 2; "FlashAttention 3 and 4: When the Bottleneck Moves", section 3.2:
 * a share of the exponentials emulated on the FMA pipe by a polynomial).
 * enable = 1: later attn_fwd / attn_fwd_gqa calls evaluate 10 of every 32
 * score columns as 2^floor(x) * p3(x - floor(x)) with the degree-3 minimax
 * polynomial on FMAs and the other 22 on the hardware ex2 unit; enable = 0
 * (the default; also the environment variable ATTN_EXP_POLY=0/1 at first use)
 * uses the hardware unit for every column.  Results meet the same tolerances
 * either way.  Returns ATTN_OK or ATTN_ERR_INVALID_ARG (enable not 0 or 1).
 */
int attn_set_exp_poly(int enable);

/*
 * Backward on CTA pairs at d = 128 ("FlashAttention-4: Algorithm and Kernel
 * Pipelining Co-Design for Asymmetric Hardware Scaling", Table 3 and Figure
 * 3: the 2-CTA backward).  With enable = 1, later attn_bwd calls with
 * d_qk = d_v = 128 run the main kernel on clusters of two CTAs: key tiles
 * 2p and 2p+1 of a head share every product (tcgen05.mma.cta_group::2,
 * M = 256, each CTA reading half of the B operand), and dQ of a query tile is
 * one pair product over both key tiles after the CTAs exchange dS halves
 * through distributed shared memory.  Results meet the same tolerances and
 * the deterministic mode stays bit-reproducible; the accumulator layout in
 * the workspace differs (workspace size unchanged).  enable = 0 (the
 * default; also the environment variable ATTN_BWD_PAIR=0/1 at first use)
 * selects the one-CTA kernel, which measures faster on GB300.  Returns
 * ATTN_OK or ATTN_ERR_INVALID_ARG (enable not 0 or 1).
 */
int attn_set_bwd_pair(int enable);

/*
 * Forward kernel selection for later attn_fwd, attn_fwd_gqa, attn_fwd_fp8 and
 * attn_fwd_masked calls: mode = 1 runs the persistent kernel (as many CTAs as
 * fit on the GPU at once, each taking units of query tiles in turn), 0 one
 * CTA per unit, -1 (the default; also ATTN_FWD_PERSIST at first use) chooses
 * by size: persistent for N <= 2048, causal N <= 4096, and windows short
 * enough to make units short (attn_fwd_masked).  Results meet the same
 * tolerances either way.  Returns ATTN_OK or ATTN_ERR_INVALID_ARG.
 */
int attn_set_fwd_persist(int mode);

/*
 * Backward main kernel selection for later attn_bwd / attn_bwd_noalloc calls:
 * mode = 1 runs the persistent kernel (one CTA per SM taking the (head, key
 * tile) units in rounds), 0 the kernel with one CTA per unit, -1 (the
 * default; also ATTN_BWD_PERSIST at first use) chooses: persistent in atomic
 * mode at every N, and in deterministic mode for N <= 2048.  Results meet the same
 * tolerances either way; deterministic mode is bit-identical run to run with
 * either kernel (the two may differ from each other in the last bits).
 * Applies to d_qk = d_v = 64 and 128 without grouped-query heads or masks;
 * the other backward calls always run one CTA per unit.  At d = 128 the
 * CTA-pair setting (attn_set_bwd_pair(1)) takes precedence: with it on, the
 * pair kernel runs whatever this mode says.  In deterministic mode the
 * persistent kernel is launched cooperatively (all its CTAs resident at once,
 * which its cross-CTA ordering of the dQ additions needs, even while other
 * kernels share the GPU).
 * Returns ATTN_OK or ATTN_ERR_INVALID_ARG.
 */
int attn_set_bwd_persist(int mode);

/*
 * Order of the work in the deterministic backward ("FlashAttention-4:
 * Algorithm and Kernel Pipelining Co-Design for Asymmetric Hardware
 * Scaling", Figures 7 and 8: the schedule ablations of the deterministic
 * backward -- head swizzle, shortest- or longest-first, reverse m-block
 * order).  The (head, key tile) units run key-tile-major inside groups of
 * ``head_group`` heads (0, the default, picks the fastest order measured on
 * GB300: without a causal mask, on the persistent kernel groups of one head
 * for N <= 2048 and one group of all heads above, on the one-unit kernel
 * one group of all heads for N <= 2048 and groups of 8 heads above; under
 * the causal mask one group of all heads; also ATTN_DET_GROUP at first use);
 * ``descending`` = 1 (ATTN_DET_DESC) takes the
 * key tiles from the last down -- shortest first under the causal mask --
 * and every dQ tile then adds its key-tile contributions in that same
 * descending order, 0 ascending (longest first under the causal mask).
 * The one-unit kernel and the causal mask visit the query tiles from the last
 * down; the persistent kernel without the causal mask (the default for
 * N <= 2048) rotates each round's walks so that
 * a head's units start at different query tiles, and a dQ tile takes the
 * additions of a round in the order of their visits (attn_bwd_det_plan
 * writes the plan out).  Each setting is
 * bit-reproducible on its own; different settings add in different orders
 * and may differ from each other in the last bits.  Applies to later
 * deterministic attn_bwd / attn_bwd_gqa / attn_bwd_noalloc calls except the
 * CTA-pair kernel (masked calls always take the default).  Returns ATTN_OK
 * or ATTN_ERR_INVALID_ARG (head_group < 0, descending not 0 or 1).
 */
int attn_set_det_schedule(int head_group, int descending);

/*
 * The deterministic backward's plan, as its kernels compute it, written out
 * for host-side checks (no GPU work).  For n_heads heads of n_tiles 128-row
 * tiles taken by n_ctas persistent CTAs in units of head_group heads
 * (clipped to n_heads) and the order ``descending`` (attn_set_det_schedule):
 * unit u (0 .. n_heads * n_tiles - 1, the launch / round order) is key tile
 * unit_key_tile[u] of head unit_head[u]; it visits the query tiles from
 * unit_first_tile[u] downwards, wrapping from 0 to n_tiles - 1 (rotated) or
 * ending at 0 (the key tile under the causal mask); and its addition to dQ
 * tile i goes ahead when that tile's ticket reaches rank[u * n_tiles + i]
 * (-1: the unit does not touch tile i).  ``rotated`` = 1 gives the walk of
 * the persistent non-causal kernel (every CTA resident at once): in each
 * round of n_ctas units the units of one head start at different query
 * tiles ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
 * Asymmetric Hardware Scaling", Figures 7-8, on the deterministic schedule).
 * Arrays are caller-owned host memory of n_heads * n_tiles ints (rank:
 * n_heads * n_tiles * n_tiles).  Returns ATTN_OK or ATTN_ERR_INVALID_ARG
 * (sizes < 1, flags not 0/1, rotated with causal, null arrays, more than
 * 2^28 ranks).
 */
int attn_bwd_det_plan(int n_heads, int n_tiles, int n_ctas, int head_group, int descending, int causal, int rotated,
                      int* unit_head, int* unit_key_tile, int* unit_first_tile, int* rank);

/*
 * Per-kernel timing for benchmarks.  Between attn_profile_start and
 * attn_profile_stop, every attn_fwd / attn_bwd call on any stream also records
 * CUDA events immediately before and after each of its kernel launches, on
 * the launch stream.  attn_profile_stop synchronises those events and fills
 * ``out`` with the launch counts and summed durations (milliseconds) per
 * kernel: the forward kernel, the backward's preprocess, main and dQ
 * conversion kernels, and attn_fwd_splitkv's forward and merge kernels (whose
 * merge then launches as an ordinary kernel rather than a programmatic
 * dependent).  Profiling adds host work per call; leave it off
 * otherwise.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG (null out / not started)
 * or ATTN_ERR_CUDA.
 */
typedef struct {
  int launches_fwd, launches_bwd_pre, launches_bwd_main, launches_bwd_convert;
  float ms_fwd, ms_bwd_pre, ms_bwd_main, ms_bwd_convert;
  int launches_fwd_split, launches_merge; /* attn_fwd_splitkv's two kernels */
  float ms_fwd_split, ms_merge;
} attn_kernel_times_t;

int attn_profile_start(void);
int attn_profile_stop(attn_kernel_times_t* out);

/*
 * Self-test of the kernels' bounded waits: launches one thread that waits on
 * a pipeline barrier nothing will complete, with a limit of ``timeout_us``
 * microseconds (1 .. 10^7).  The wait gives up, the kernel records
 * ATTN_ERR_TIMEOUT in the device status word and returns, and the context
 * stays usable; attn_get_device_status then reports it (where = 900).
 */
int attn_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream);

/*
 * Size of the device array attn_bwd_noalloc uses as its workspace: 32 MiB on
 * every GPU that loads this library, held until the process exits.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * attn_bwd without a caller-provided workspace.  The pages describe no such
 * call (it has no counterpart in the paper): it exists for callers that
 * cannot allocate device memory -- code running in a host callback, or inside
 * a runtime that hands out every device buffer itself and forbids
 * allocations on its request path -- and so cannot supply attn_bwd's
 * workspace.  The workspace is a static device array of
 * ATTN_NOALLOC_SCRATCH_BYTES inside the library; nothing is allocated.
 *   Arguments, layouts and results are those of attn_bwd without
 *   ``workspace`` / ``workspace_bytes``.
 *   Sizes whose workspace does not fit ATTN_NOALLOC_SCRATCH_BYTES return
 *   ATTN_ERR_WORKSPACE, other argument errors as attn_bwd.  When only the
 *   persistent kernel's region for cut units (see attn_bwd_workspace_bytes)
 *   does not fit, the call runs without it: that kernel's last round then
 *   takes whole units.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 *   All calls on a device share the array: calls whose kernels can overlap on
 *   the GPU (unordered streams) race and give wrong results.  Each call
 *   clears what it needs at its start, so back-to-back calls are correct.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                     void* dq, void* dk, void* dv, int B, int H, int N, int d_qk, int d_v, int causal, float scale,
                     int deterministic, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
