/*
 * spec_control.h — C ABI of the draft-length controller in libspecverify.so: host-side
 * acceptance statistics over verified batches and the number of drafts K for the next batch.
 *
 * What it follows (cited as host + section of the page):
 *   - 2kiu.com/news/5895634 §4.4: keep a sliding window of per-batch acceptance rates; when the
 *     mean over the last 100 batches is above 0.8 raise K by one, when it is below 0.6 lower K by
 *     one, and keep K within [2, 10]; when many recent batches accept poorly, switch
 *     speculation off for a while and switch it back on once acceptance recovers;
 *   - 2kiu.com/news/5895634 §7: the switch-off threshold is a windowed acceptance rate below 0.5;
 *   - cf-1.com/news/5155685 §2.4: the draft length follows the recent acceptance history.
 * Readings where the pages are silent (the controller's defaults are the pages' numbers):
 *   - a batch's acceptance rate is sum_b n_acc_b / sum_b K_b over its requests (accepted drafts
 *     per proposed draft); a batch that proposed no draft adds nothing to the window;
 *   - the window mean is the plain mean of the last `window` batch rates, and a decision is taken
 *     only on a full window; after any change of K the window starts empty, so every decision
 *     rests on `window` batches run at the current K;
 *   - thresholds are strict and compared in float (the mean rounded to float): raise when
 *     mean > raise_above, lower when mean < lower_below, switch off when mean < disable_below
 *     (checked first);
 *   - with speculation off nothing measures acceptance, so after `probe_after` batches decoded
 *     without drafts the controller probes again at K = k_min with an empty window.
 *
 * Conventions: all pointers are host memory; a controller is not thread-safe (one per scheduler
 * thread); the library allocates the controller in spec_ctrl_create and frees it in
 * spec_ctrl_destroy, nothing else.  No function touches the GPU.
 */
#ifndef SPEC_CONTROL_H_
#define SPEC_CONTROL_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t k_init;        /* K of the first batch (clamped into [k_min, k_max])             */
  int32_t k_min;         /* lower bound of K, >= 1 (pages: 2)                                */
  int32_t k_max;         /* upper bound of K, >= k_min, <= 64 (pages: 10)                    */
  int32_t window;        /* batches in the sliding window, 1..100000 (pages: 100)            */
  float raise_above;     /* raise K when the window mean exceeds this (pages: 0.8)           */
  float lower_below;     /* lower K when the window mean is below this (pages: 0.6)          */
  float disable_below;   /* switch speculation off below this (pages: 0.5); 0 = never        */
  int32_t probe_after;   /* batches without drafts before probing again at k_min, >= 1      */
} spec_ctrl_config_t;

typedef struct spec_ctrl spec_ctrl_t; /* opaque */

/* The pages' settings: k_init 4, k_min 2, k_max 10, window 100, 0.8 / 0.6 / 0.5, probe after 100. */
void spec_ctrl_default_config(spec_ctrl_config_t* cfg);

/* A controller for `cfg` (copied), or NULL if cfg is NULL or out of range
 * (requires disable_below <= lower_below < raise_above <= 1). */
spec_ctrl_t* spec_ctrl_create(const spec_ctrl_config_t* cfg);

void spec_ctrl_destroy(spec_ctrl_t* ctrl);

/*
 * Record one verified batch and return the K for the next batch (0 = speculation off: decode
 * the next batch without drafts and report it with spec_ctrl_skip).
 *   num_accepted [B] int32: out_num_accepted of the verify step;
 *   k_per_row [B] int32 or NULL: the drafts each request proposed (NULL = K_used for all);
 *   K_used: the K the batch ran with.
 * Entries of k_per_row are clamped into [0, K_used] and num_accepted into [0, K_b], as the
 * verify step clamps them.  Returns -1 for a NULL controller or B < 0 (nothing recorded).
 */
int32_t spec_ctrl_update(spec_ctrl_t* ctrl, const int32_t* num_accepted, const int32_t* k_per_row,
                         int32_t B, int32_t K_used);

/* Record one batch decoded without drafts; returns the K for the next batch (0 while off). */
int32_t spec_ctrl_skip(spec_ctrl_t* ctrl);

/* The K the next batch should use (0 = off), or -1 for a NULL controller. */
int32_t spec_ctrl_k(const spec_ctrl_t* ctrl);

/* Mean of the batch rates in the window so far (NaN when empty), and how many it holds. */
double spec_ctrl_window_mean(const spec_ctrl_t* ctrl);
int32_t spec_ctrl_window_fill(const spec_ctrl_t* ctrl);

/* Totals since creation: accepted drafts, proposed drafts, verified batches. */
void spec_ctrl_totals(const spec_ctrl_t* ctrl, int64_t* accepted, int64_t* proposed, int64_t* batches);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_CONTROL_H_ */
