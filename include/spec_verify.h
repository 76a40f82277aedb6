/*
 * spec_verify.h — C ABI of libspecverify.so: the verify step of speculative sampling on one GPU.
 *
 * What the step computes (cited as host + section of the page that defines it):
 *   - cf-1.com/news/5155685 §2.2 and 2kiu.com/news/5895634 §2.2: a draft token x drawn from the
 *     draft distribution q is accepted with probability min(1, p(x)/q(x)); on rejection a token is
 *     drawn from norm(max(0, p - q)), so the emitted token is distributed as p;
 *   - cf-1.com/news/5155685 §2.1 and gsyq.cn/news/428210 §3.1: positions are judged in order and
 *     the output is cut at the first rejected position;
 *   - gsyq.cn/news/428210 §3.2 and 2kiu.com/news/5895634 §3.1: one target forward yields
 *     1 + a + ... + a^K tokens on average, i.e. when every draft is accepted one more token is
 *     drawn from p at position K (the bonus token);
 *   - gsyq.cn/news/428210 §3.3: temperature, top-k and top-p are shared sampling parameters of
 *     both sides; 2kiu.com/news/5895634 §7: the draft may sample at its own temperature.
 * Readings where the pages are silent: temperature divides both logit sets; top-k keeps every
 * logit >= the k-th largest (ties kept and flagged); accept iff u * q(x) < p(x); the inverse CDF
 * runs in ascending token id with the strict rule u * R < C_v; temperature 0 is the greedy limit
 * (accept iff x == argmax p, lowest index on ties; the emitted token is that argmax).
 *
 * Conventions for every entry point:
 *   - Device pointers are caller-owned device memory; the library never allocates, frees or
 *     synchronises (spec_verify_host is the one exception: it synchronises its stream).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and is
 *     asynchronous with respect to the host.
 *   - The return code covers what the host can check.  Data-dependent problems (a draft token
 *     outside [0, V), k_per_row outside [0, K_max], NaN / +inf logits, rounding fallbacks) are
 *     reported per request in stats.flags and never trap.
 *   - The library keeps no per-call global state and is safe to call from several host threads
 *     on distinct workspaces.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPEC_DTYPE_F32 = 0, SPEC_DTYPE_BF16 = 1 } spec_dtype_t;

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* a null required pointer, a negative size, T < 0, top_k < 0, ...  */
  SPEC_ERR_UNSUPPORTED = 2, /* sizes beyond the limits below, or an unknown dtype              */
  SPEC_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, copy, attribute query)       */
  SPEC_ERR_WORKSPACE = 4,   /* workspace NULL, misaligned (< 256 B) or smaller than required    */
  SPEC_ERR_TIMEOUT = 5      /* reserved: no kernel of this library waits on another block       */
} spec_status_t;

/* Per-request flag bits of spec_verify_stats_t.flags. */
#define SPEC_FLAG_RESIDUAL_ZERO 1 /* max(0, p - q) summed to 0 after rounding: drew from p   */
#define SPEC_FLAG_CDF_CLAMP 2     /* u * R fell past the last cumulative sum: took the last v  */
#define SPEC_FLAG_BAD_TOKEN 4     /* a draft token outside [0, V): treated as p = q = 0        */
#define SPEC_FLAG_BAD_K 8         /* k_per_row outside [0, K_max]: clamped into range          */
#define SPEC_FLAG_NONFINITE 16    /* a NaN / +inf logit or an all -inf row: result unspecified */
#define SPEC_FLAG_TOPK_TIE 32     /* top-k kept more than k logits of some row (ties)          */

/* Limits (SPEC_ERR_UNSUPPORTED beyond them). */
#define SPEC_MAX_K 16        /* K_max                                                        */
#define SPEC_MAX_V 2097152   /* vocabulary size                                              */
#define SPEC_MAX_TOPK 256    /* top_k values in (0, V) above this take SPEC_ERR_UNSUPPORTED   */
#define SPEC_MAX_DRAFTS 4    /* draft chains per request of spec_verify_multi                 */

/*
 * Optional diagnostics.  Every pointer is device memory and may be NULL (= not written).
 *   p_draft, q_draft [B * K_max] float: normalised p_j(x_j), q_j(x_j) at the examined positions
 *       (j <= first rejection), NaN elsewhere and in greedy mode;
 *   accept_margin [B * K_max] float: |u_j - p_j(x_j)/q_j(x_j)| (inf when q_j(x_j) == 0), NaN where
 *       p_draft is NaN; a decision with margin < 1e-5 may legitimately differ from an fp64 oracle;
 *   sample_margin [B] float: distance of u_resample to the nearer edge of the drawn token's CDF
 *       interval (inf in greedy mode);
 *   residual_mass [B] float: sum_v max(0, p - q) at the first rejected position, 0 for a bonus draw;
 *   row_lognorm [B * (2*K_max + 1)] float: per row, max(z)/T + ln sum_v exp((z_v - max z)/T) over
 *       the kept set; p rows 0..K_max then q rows 0..K_max-1; NaN for rows past K_b and in greedy mode;
 *   flags [B] int32: SPEC_FLAG_* bits;
 *   pass1_done: a cudaEvent_t (host handle, cast to void*) recorded on the stream between the
 *       streaming pass and the per-request pass, so a caller can time the two passes apart; NULL
 *       = not recorded.  It is the one field that is not device memory;
 *   row_cut [B * (2*K_max + 1)] float: per row (same order as row_lognorm), the smallest logit the
 *       row keeps: the top-k threshold (the k-th largest logit) or the nucleus cut (the logit of the
 *       last tie group kept), whichever is larger; -inf when neither truncation is on; NaN for rows
 *       past K_b and in greedy mode.  The kept set of a row is {v : z_v >= row_cut}.
 */
typedef struct {
  float* p_draft;
  float* q_draft;
  float* accept_margin;
  float* sample_margin;
  float* residual_mass;
  float* row_lognorm;
  int32_t* flags;
  void* pass1_done;
  float* row_cut;
} spec_verify_stats_t;

/*
 * Bytes of device workspace spec_verify needs for these sizes, for any temperature (0 for invalid
 * sizes).  The workspace holds per-call scratch only (per-chunk summaries, top-k candidates, the
 * ragged row table): it needs no initialisation and keeps nothing between calls, but one
 * workspace must not be used by two calls that may run at the same time.
 */
size_t spec_verify_workspace_bytes(int32_t B, int32_t K_max, int32_t V, spec_dtype_t dtype,
                                   int32_t top_k);

/*
 * The verify step for a batch of B independent requests (all pointers device memory):
 *   p_logits      [B, K_max+1, V] dtype: target logits, position K_b is the bonus position;
 *   q_logits      [B, K_max, V] dtype: draft logits (may be NULL iff temperature == 0);
 *   draft_tokens  [B, K_max] int32: x_0..x_{K_b-1} (entries past K_b are not read);
 *   k_per_row     [B] int32 or NULL: K_b in [0, K_max] drafts of request b (NULL: all K_max);
 *                 rows past K_b are never read, so ragged batches use the padded layout;
 *   u_accept      [B, K_max] float in [0, 1): one uniform per (request, position) (NULL iff T == 0);
 *   u_resample    [B] float in [0, 1): one uniform per request for the resample or bonus draw
 *                 (NULL iff T == 0);
 *   temperature   > 0, or 0 for greedy argmax-match;
 *   top_k         0 = off, >= V = off, else keep the top_k largest logits of every row (<= 256);
 *   out_tokens    [B, K_max+1] int32: x_0..x_{n-1}, then the resampled / bonus / argmax token,
 *                 then -1 padding;
 *   out_num_accepted [B] int32: n = accepted drafts, in [0, K_b];
 *   out_stats     host struct of device pointers, or NULL;
 *   workspace     device memory of at least spec_verify_workspace_bytes(...) bytes, 256-B aligned.
 * Launches two kernels (three with k_per_row): a streaming pass over every valid logit row that
 * leaves per-chunk summaries in the workspace, then the per-request pass for the decision and the
 * draw (one block per request; a cluster of 8 blocks per request when the batch has fewer requests
 * than the GPU has SMs and the rows are long).  Returns SPEC_OK once the work is enqueued.
 */
spec_status_t spec_verify(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                          const int32_t* k_per_row, const float* u_accept, const float* u_resample,
                          float temperature, int32_t top_k, int32_t* out_tokens,
                          int32_t* out_num_accepted, const spec_verify_stats_t* out_stats, int32_t B,
                          int32_t K_max, int32_t V, spec_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Sampling parameters of spec_verify_ex.
 *   temperature        T of the target rows: > 0, or 0 for greedy argmax-match (then the other
 *                      fields are not used);
 *   draft_temperature  T_q the draft sampled its tokens with (2kiu.com/news/5895634 §7: the draft
 *                      may run cooler than the target); > 0; the q rows are divided by it;
 *   top_k              as for spec_verify (0 or >= V = off, else <= SPEC_MAX_TOPK);
 *   top_p              nucleus mass in (0, 1]; >= 1 = off (gsyq.cn/news/428210 §3.3 names top_p
 *                      among the parameters draft and target must share).  After temperature and
 *                      top-k, every row keeps the smallest set of most likely tokens whose mass
 *                      reaches top_p, with every token tied with the last one, and is
 *                      renormalised.  The cut compares fp32 sums with top_p: where the cumulative
 *                      mass lies within ~1e-6 of top_p the kept set may differ from an exact one.
 */
typedef struct {
  float temperature;
  float draft_temperature;
  int32_t top_k;
  float top_p;
} spec_sampling_t;

/*
 * spec_verify with the sampling parameters of spec_sampling_t (all other arguments, the
 * workspace size and the results as for spec_verify; `sampling` is a host pointer read before
 * the call returns).  spec_verify(..., T, top_k, ...) is spec_verify_ex with {T, T, top_k, 1}.
 * With top_p < 1 (and top-k off) a nucleus pass between the two reads every valid row once more to
 * find its nucleus: twice when the cut lies below 2^-13 of the max's weight, and a few times more
 * (4-bit key digits, mostly from L2) for rows whose head is crowded or whose cut lies below 2^-15.
 * After top-k the per-request pass finds the nucleus among the kept candidates.
 * Returns SPEC_ERR_INVALID_ARG for sampling == NULL, T_q <= 0 with T > 0, or top_p <= 0 / NaN.
 */
spec_status_t spec_verify_ex(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                             const int32_t* k_per_row, const float* u_accept, const float* u_resample,
                             const spec_sampling_t* sampling, int32_t* out_tokens,
                             int32_t* out_num_accepted, const spec_verify_stats_t* out_stats, int32_t B,
                             int32_t K_max, int32_t V, spec_dtype_t dtype, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * Device bytes spec_verify_host needs as staging for these sizes (inputs, outputs and the
 * spec_verify workspace, each 256-B aligned), or 0 for invalid sizes.
 */
size_t spec_verify_host_staging_bytes(int32_t B, int32_t K_max, int32_t V, spec_dtype_t dtype,
                                      int32_t top_k, int32_t has_k_per_row);

/*
 * The same step on HOST buffers: copies the inputs into `staging` (device memory of at least
 * spec_verify_host_staging_bytes(...) bytes, no initialisation needed), runs spec_verify there,
 * copies out_tokens and
 * out_num_accepted back, and synchronises `stream` before returning.  Host pointers follow the
 * layouts of spec_verify; q_logits / u_accept / u_resample may be NULL iff temperature == 0 and
 * k_per_row may be NULL.  Pinned (page-locked) host memory makes the copies asynchronous DMA.
 */
spec_status_t spec_verify_host(const void* p_logits, const void* q_logits,
                               const int32_t* draft_tokens, const int32_t* k_per_row,
                               const float* u_accept, const float* u_resample, float temperature,
                               int32_t top_k, int32_t* out_tokens, int32_t* out_num_accepted,
                               int32_t B, int32_t K_max, int32_t V, spec_dtype_t dtype,
                               void* staging, size_t staging_bytes, void* stream);

/*
 * spec_verify_host with the sampling parameters of spec_sampling_t (staging size as for
 * spec_verify_host; spec_verify_host(..., T, top_k, ...) is this call with {T, T, top_k, 1}).
 */
spec_status_t spec_verify_host_ex(const void* p_logits, const void* q_logits,
                                  const int32_t* draft_tokens, const int32_t* k_per_row,
                                  const float* u_accept, const float* u_resample,
                                  const spec_sampling_t* sampling, int32_t* out_tokens,
                                  int32_t* out_num_accepted, int32_t B, int32_t K_max, int32_t V,
                                  spec_dtype_t dtype, void* staging, size_t staging_bytes, void* stream);

/*
 * Draft-token sampling, the step before verification (gsyq.cn/news/428210 §3.1: the draft model
 * proposes its tokens by sampling its own distribution): one token per row of `logits`, drawn
 * from the row's distribution after temperature, top-k and top-p by the same inverse CDF as the
 * verify step's bonus draw: x = the smallest v with u * S < C_v, C_v cumulative in ascending
 * token id over the kept set (greedy argmax, lowest index, at temperature 0).  It is
 * spec_verify_ex on a batch of `rows` requests with no drafts.
 *   logits [rows, V] dtype (device); u [rows] float in [0, 1) (device; NULL iff temperature == 0);
 *   sampling: temperature, top_k, top_p (draft_temperature is not used);
 *   out_tokens [rows] int32 (device): the drawn token, -1 for a row with NaN / +inf logits;
 *   out_prob [rows] float (device) or NULL: the drawn token's probability q(x) under that
 *       distribution (1 in greedy mode, NaN where out_tokens is -1);
 *   workspace: spec_sample_workspace_bytes(...) bytes of device memory, 256-B aligned.
 * Errors as for spec_verify_ex.
 */
size_t spec_sample_workspace_bytes(int32_t rows, int32_t V, spec_dtype_t dtype, int32_t top_k);
spec_status_t spec_sample(const void* logits, const float* u, const spec_sampling_t* sampling, int32_t* out_tokens,
                          float* out_prob, int32_t rows, int32_t V, spec_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Multi-draft verify: N draft chains per request (2kiu.com/news/5895634 §7 and cf-1.com/news/5155685
 * §2.3 name ensembles of draft models whose accepted draft the target keeps).  The pages fix the
 * property the step keeps -- the emitted tokens are distributed as p (cf-1.com §2.2, 2kiu.com §2.2) --
 * but no rule for several candidates; the rule here tests the chains' first drafts in turn, each
 * against what the earlier rejections leave of p:
 *   r_0 = P_0; candidate n (first draft x_n of chain n, drawn from its draft distribution Q_n) is
 *   accepted iff u_n * Q_n(x_n) < r_n(x_n); a rejection leaves r_{n+1} = norm(max(0, r_n - Q_n));
 *   the first accepted chain is verified on with the single-draft rule (as spec_verify) on its own
 *   rows; with every candidate rejected one token is drawn from r_N (inverse CDF, ascending token
 *   id, u_resample).  Temperature 0: the first chain whose first draft is the argmax of P_0 (lowest
 *   index on ties) is followed with the greedy rule; none: the argmax is emitted.
 *   p_logits      [B, N, K_max+1, V] dtype: the target's logits along each chain; row 0 of chain 0
 *                 is the shared first position (row 0 of the other chains is never read);
 *   q_logits      [B, N, K_max, V] dtype: each chain's draft logits (NULL iff temperature == 0);
 *   draft_tokens  [B, N, K_max] int32;  u_accept [B, N, K_max] float (NULL iff temperature == 0):
 *                 u_accept[b, n, 0] tests candidate n, u_accept[b, n, j] position j of chain n;
 *   u_resample    [B] float (NULL iff temperature == 0);
 *   sampling      temperature and draft_temperature as for spec_verify_ex; top_k must be off and
 *                 top_p >= 1 (SPEC_ERR_UNSUPPORTED otherwise);
 *   out_tokens    [B, K_max+1] int32: the emitted tokens, then -1;  out_num_accepted [B] int32;
 *   out_chain     [B] int32 or NULL: the accepted chain, -1 when every candidate was rejected;
 *   out_flags     [B] int32 or NULL: SPEC_FLAG_* bits (a non-finite row anywhere in a request leaves
 *                 it without a result: n_acc 0, tokens -1, chain -1);
 *   workspace     spec_verify_multi_workspace_bytes(...) bytes of device memory, 256-B aligned.
 * Every chain has K_max drafts (no k_per_row).  1 <= N <= SPEC_MAX_DRAFTS.  With N = 1 the rule is
 * spec_verify's (the draws' sums may round differently).  Launches the row table, the streaming pass
 * over every row read, and the per-request pass (a cluster of 4 blocks per request when sampling,
 * one block when greedy); asynchronous on `stream`.
 */
size_t spec_verify_multi_workspace_bytes(int32_t B, int32_t N, int32_t K_max, int32_t V, spec_dtype_t dtype);
spec_status_t spec_verify_multi(const void* p_logits, const void* q_logits, const int32_t* draft_tokens,
                                const float* u_accept, const float* u_resample, const spec_sampling_t* sampling,
                                int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_chain,
                                int32_t* out_flags, int32_t B, int32_t N, int32_t K_max, int32_t V,
                                spec_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Test support, not for production use.  With bit 0 of `hooks` set, every later call (from any
 * host thread) makes each block of the streaming pass treat the chunks it was to read as lost:
 * it leaves their summaries NaN, as a failed load would, instead of reading them, and every
 * request of a batch in sampling or greedy mode over 16-byte-aligned rows comes out with
 * SPEC_FLAG_NONFINITE, n_acc 0 and tokens -1 (top-k batches and unaligned rows are not
 * affected).  It exercises the handling of a lost streaming item without any fault.  0 restores
 * normal operation.
 */
void spec_verify_set_test_hooks(int32_t hooks);

/* Size of the fixed device array behind spec_verify_static (16 MiB). */
#define SPEC_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * spec_verify without a workspace argument, for callers that cannot allocate device memory: a
 * custom operator running inside a framework whose memory pool owns every allocation, or a loop
 * that must never block on cudaMalloc / cudaFree.  (This entry point has no counterpart in the
 * pages; it only changes where the scratch lives.)
 *   - The scratch is one file-scope device array of SPEC_STATIC_SCRATCH_BYTES that every GPU
 *     loading this library keeps until the process exits; it needs no initialisation.
 *   - The first call on a device (the current device) looks up the array's device address with
 *     cudaGetSymbolAddress and caches it; make that first call before any stream capture.
 *   - Arguments are checked as spec_verify checks them, with the same status codes; then a call
 *     whose own workspace (for its mode -- sampling, top-k or greedy -- and its row layout) exceeds
 *     the array is rejected with SPEC_ERR_WORKSPACE before anything is launched.  For example
 *     B=1024, K_max=4, V=128256 fits in bf16 (about 9.5 MB) and in greedy fp32 (about 10.5 MB), but
 *     not in sampled fp32 (about 19 MB); large top-k batches do not fit.
 *   - Every call on a device shares the one array: calls that may overlap on the GPU (other
 *     streams, other host threads) race and corrupt each other; serialise them.
 *   - Allocates nothing; all other arguments and results are as for spec_verify.
 */
spec_status_t spec_verify_static(const void* p_logits, const void* q_logits,
                                 const int32_t* draft_tokens, const int32_t* k_per_row,
                                 const float* u_accept, const float* u_resample, float temperature,
                                 int32_t top_k, int32_t* out_tokens, int32_t* out_num_accepted,
                                 const spec_verify_stats_t* out_stats, int32_t B, int32_t K_max,
                                 int32_t V, spec_dtype_t dtype, void* stream);

/* A static, human-readable name for a status code. */
const char* spec_verify_status_string(spec_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
