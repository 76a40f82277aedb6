// spec_control.cpp — the draft-length controller declared in spec_control.h: a sliding window of
// per-batch acceptance rates drives K up or down by one within [k_min, k_max], and a poor window
// switches speculation off until a later probe (2kiu.com/news/5895634 §4.4 and §7,
// cf-1.com/news/5155685 §2.4).  Host code only.
#include "spec_control.h"

#include <cmath>
#include <cstdint>
#include <new>
#include <vector>

struct spec_ctrl {
  spec_ctrl_config_t cfg;
  int32_t k;               // K of the next batch; 0 while speculation is off
  std::vector<double> ring;  // the window's batch rates
  int32_t head = 0;        // next slot of the ring
  int32_t fill = 0;        // rates held
  int32_t off_batches = 0;
  int64_t accepted = 0, proposed = 0, batches = 0;
};

namespace {

int32_t clampi(int32_t x, int32_t lo, int32_t hi) { return x < lo ? lo : (x > hi ? hi : x); }

void clear_window(spec_ctrl* c) {
  c->head = 0;
  c->fill = 0;
}

void push_rate(spec_ctrl* c, double r) {
  const int32_t w = c->cfg.window;
  if (c->fill < w) ++c->fill;
  c->ring[c->head] = r;
  c->head = c->head + 1 == w ? 0 : c->head + 1;
}

// The mean of the window, summed afresh from the ring (slots 0..fill-1 hold it).
double window_mean(const spec_ctrl* c) {
  if (c->fill == 0) return NAN;
  double s = 0.0;
  for (int32_t i = 0; i < c->fill; ++i) s += c->ring[i];
  return s / c->fill;
}

void decide(spec_ctrl* c) {
  if (c->fill < c->cfg.window) return;  // decisions rest on a full window
  // compared in the thresholds' own precision, so a mean of exactly 0.6 is not "below 0.6f"
  const float m = (float)window_mean(c);
  if (m < c->cfg.disable_below) {
    c->k = 0;
    c->off_batches = 0;
    clear_window(c);
  } else if (m > c->cfg.raise_above && c->k < c->cfg.k_max) {
    ++c->k;
    clear_window(c);
  } else if (m < c->cfg.lower_below && c->k > c->cfg.k_min) {
    --c->k;
    clear_window(c);
  }
}

}  // namespace

extern "C" {

void spec_ctrl_default_config(spec_ctrl_config_t* cfg) {
  if (!cfg) return;
  cfg->k_init = 4;
  cfg->k_min = 2;
  cfg->k_max = 10;
  cfg->window = 100;
  cfg->raise_above = 0.8f;
  cfg->lower_below = 0.6f;
  cfg->disable_below = 0.5f;
  cfg->probe_after = 100;
}

spec_ctrl_t* spec_ctrl_create(const spec_ctrl_config_t* cfg) {
  if (!cfg) return nullptr;
  const spec_ctrl_config_t& g = *cfg;
  if (g.k_min < 1 || g.k_max < g.k_min || g.k_max > 64) return nullptr;
  if (g.window < 1 || g.window > 100000 || g.probe_after < 1) return nullptr;
  if (!(g.disable_below >= 0.0f) || !(g.disable_below <= g.lower_below) || !(g.lower_below < g.raise_above) ||
      !(g.raise_above <= 1.0f))
    return nullptr;
  spec_ctrl* c = new (std::nothrow) spec_ctrl;
  if (!c) return nullptr;
  c->cfg = g;
  c->k = clampi(g.k_init, g.k_min, g.k_max);
  c->ring.assign((size_t)g.window, 0.0);
  return c;
}

void spec_ctrl_destroy(spec_ctrl_t* ctrl) { delete ctrl; }

int32_t spec_ctrl_update(spec_ctrl_t* c, const int32_t* num_accepted, const int32_t* k_per_row, int32_t B,
                         int32_t K_used) {
  if (!c || B < 0 || (B > 0 && !num_accepted)) return -1;
  if (K_used < 0) K_used = 0;
  int64_t acc = 0, prop = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t kb = k_per_row ? clampi(k_per_row[b], 0, K_used) : K_used;
    acc += clampi(num_accepted[b], 0, kb);
    prop += kb;
  }
  c->accepted += acc;
  c->proposed += prop;
  ++c->batches;
  if (prop > 0) {
    push_rate(c, (double)acc / (double)prop);
    if (c->k > 0) decide(c);
  }
  return c->k;
}

int32_t spec_ctrl_skip(spec_ctrl_t* c) {
  if (!c) return -1;
  if (c->k == 0 && ++c->off_batches >= c->cfg.probe_after) {
    c->k = c->cfg.k_min;  // probe: speculate again and measure with a fresh window
    c->off_batches = 0;
    clear_window(c);
  }
  return c->k;
}

int32_t spec_ctrl_k(const spec_ctrl_t* c) { return c ? c->k : -1; }

double spec_ctrl_window_mean(const spec_ctrl_t* c) { return c ? window_mean(c) : NAN; }

int32_t spec_ctrl_window_fill(const spec_ctrl_t* c) { return c ? c->fill : -1; }

void spec_ctrl_totals(const spec_ctrl_t* c, int64_t* accepted, int64_t* proposed, int64_t* batches) {
  if (accepted) *accepted = c ? c->accepted : 0;
  if (proposed) *proposed = c ? c->proposed : 0;
  if (batches) *batches = c ? c->batches : 0;
}

}  // extern "C"
