// Host-side controller and metrics of the verify step (no GPU code).
//
// Page 3 ("推测解码的工程真相 2026"), dynamic-scheduling and observability
// sections: per request, the acceptance rate of its last 16 verify steps
// sets the next draft length (above 60%: 8 drafts, 30-60%: 4, below 30%:
// 2), a temperature above 0.8 sets it to 1 at once, and a request whose
// speculation does not pay falls back to plain decoding; the metrics to
// watch are the acceptance-rate distribution (P50/P95/P99 and a histogram
// that separates a low and a high mode), the speculative efficiency, the
// tree width effective and the fallback rate.  Page 2 §5.1: log the drafted
// and accepted counts of every step and where the rejections fall.
//
// Readings (the pages leave these open or garble them):
//   * speculative efficiency: the page's product "acceptance rate x mean
//     accepted / draft steps" never exceeds 1 and cannot separate gain from
//     loss, which the page says it does; it is read as page 2 §2.3's speedup
//     of one verify step: tokens emitted per step (accepted + 1) over the
//     cost of the step in target-forward units, 1 + gamma * c, with c the
//     draft model's cost relative to the target's (0.02 in page 2's worked
//     example).  Above 1 the speculation pays.
//   * tree width effective: of the drafted tree's root-to-leaf paths, the
//     share that contains the first accepted node (the paths the acceptance
//     "hit"), 0 when nothing was accepted.
//   * fallback rate: the share of requests the controller put back on plain
//     decoding (gamma 0), counting requests the device reported as failed
//     (accepted_len = -1, such as SPEC_ERR_CAPACITY, the pages' own fallback
//     trigger) as fallbacks too.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "../../include/spec_verify.h"

extern "C" {

void spec_ctrl_default_config(spec_ctrl_config* c) {
  if (c == nullptr) return;
  c->window = 16;
  c->high_acceptance = 0.6f;
  c->low_acceptance = 0.3f;
  c->gamma_high = 8;
  c->gamma_mid = 4;
  c->gamma_low = 2;
  c->hot_temperature = 0.8f;
  c->gamma_hot = 1;
  c->draft_cost = 0.02f;
  c->min_efficiency = 1.0f;
  c->max_gamma = 63;
}

spec_status spec_ctrl_init(spec_ctrl_request* reqs, int32_t n, int32_t gamma0) {
  if (reqs == nullptr || n < 0 || gamma0 < 0 || gamma0 > 63)
    return SPEC_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    memset(&reqs[i], 0, sizeof(spec_ctrl_request));
    reqs[i].gamma = gamma0;
  }
  return SPEC_OK;
}

static spec_status check_config(const spec_ctrl_config* c) {
  if (c == nullptr) return SPEC_ERR_INVALID_ARG;
  if (c->window < 1 || c->window > SPEC_CTRL_MAX_WINDOW) return SPEC_ERR_INVALID_ARG;
  if (!(c->low_acceptance >= 0.f && c->low_acceptance <= c->high_acceptance &&
        c->high_acceptance <= 1.f))
    return SPEC_ERR_INVALID_ARG;
  if (c->gamma_high < 0 || c->gamma_mid < 0 || c->gamma_low < 0 || c->gamma_hot < 0 ||
      c->max_gamma < 0 || c->max_gamma > 63)
    return SPEC_ERR_INVALID_ARG;
  if (!(c->draft_cost >= 0.f) || !(c->min_efficiency >= 0.f)) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

// Window sums of one request: drafted and accepted tokens, steps.
static void window_sums(const spec_ctrl_request& r, int window, double* drafted, double* accepted,
                        double* emitted, double* gamma_sum, int* steps) {
  const int n = r.steps < window ? r.steps : window;
  double dsum = 0, asum = 0, esum = 0;
  for (int k = 0; k < n; ++k) {
    const int i = (r.head - 1 - k + SPEC_CTRL_MAX_WINDOW) % SPEC_CTRL_MAX_WINDOW;
    dsum += r.drafted[i];
    asum += r.accepted[i];
    esum += r.accepted[i] + 1;
  }
  *drafted = dsum;
  *accepted = asum;
  *emitted = esum;
  *gamma_sum = dsum;
  *steps = n;
}

spec_status spec_ctrl_update(const spec_ctrl_config* cfg, spec_ctrl_request* reqs, int32_t n,
                             const int32_t* accepted_len, const float* temperature,
                             int32_t* next_gamma) {
  spec_status s = check_config(cfg);
  if (s != SPEC_OK) return s;
  if (reqs == nullptr || accepted_len == nullptr || next_gamma == nullptr || n < 0)
    return SPEC_ERR_INVALID_ARG;
  for (int b = 0; b < n; ++b) {
    spec_ctrl_request& r = reqs[b];
    const int a = accepted_len[b];
    if (r.gamma > 0) {
      if (a < 0) {
        // the device could not verify this step (capacity, bad input): plain decoding
        r.fallback = 1;
        r.gamma = 0;
        ++r.failed_steps;
        next_gamma[b] = 0;
        continue;
      }
      // the step that just ran drafted r.gamma tokens and accepted a of them
      r.drafted[r.head] = (int16_t)r.gamma;
      r.accepted[r.head] = (int16_t)(a < r.gamma ? a : r.gamma);
      r.head = (r.head + 1) % SPEC_CTRL_MAX_WINDOW;
      if (r.steps < SPEC_CTRL_MAX_WINDOW) ++r.steps;
    }
    if (r.fallback) {
      next_gamma[b] = 0;
      continue;
    }
    double dr, ac, em, gs;
    int steps;
    window_sums(r, cfg->window, &dr, &ac, &em, &gs, &steps);
    int g = r.gamma;
    const float T = temperature != nullptr ? temperature[b] : 0.f;
    if (temperature != nullptr && T > cfg->hot_temperature) {
      g = cfg->gamma_hot;  // draft and target laws drift apart at high temperature
    } else if (steps > 0 && dr > 0) {
      // compared in single precision, as the thresholds are given
      const float rate = (float)(ac / dr);
      g = rate > cfg->high_acceptance ? cfg->gamma_high
          : rate >= cfg->low_acceptance ? cfg->gamma_mid
                                        : cfg->gamma_low;
    }
    // a full window whose speculation does not pay: plain decoding
    if (steps >= cfg->window && dr > 0) {
      const double eff = (em / steps) / (1.0 + (gs / steps) * cfg->draft_cost);
      if (eff < cfg->min_efficiency) {
        r.fallback = 1;
        g = 0;
      }
    }
    if (g > cfg->max_gamma) g = cfg->max_gamma;
    r.gamma = g;
    next_gamma[b] = g;
  }
  return SPEC_OK;
}

spec_status spec_ctrl_metrics(const spec_ctrl_config* cfg, const spec_ctrl_request* reqs,
                              int32_t n, spec_ctrl_metrics_out* out) {
  spec_status s = check_config(cfg);
  if (s != SPEC_OK) return s;
  if (reqs == nullptr || out == nullptr || n < 0) return SPEC_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  std::vector<double> rates;
  double em_total = 0, steps_total = 0, gamma_total = 0;
  int fallbacks = 0;
  for (int b = 0; b < n; ++b) {
    const spec_ctrl_request& r = reqs[b];
    if (r.fallback) ++fallbacks;
    double dr, ac, em, gs;
    int steps;
    window_sums(r, cfg->window, &dr, &ac, &em, &gs, &steps);
    if (steps == 0 || dr <= 0) continue;
    const double rate = ac / dr;
    rates.push_back(rate);
    int bin = (int)(rate * SPEC_CTRL_HIST_BINS);
    if (bin >= SPEC_CTRL_HIST_BINS) bin = SPEC_CTRL_HIST_BINS - 1;
    ++out->acceptance_hist[bin];
    em_total += em;
    steps_total += steps;
    gamma_total += gs;
  }
  out->requests = n;
  out->fallback_rate = n > 0 ? (float)fallbacks / (float)n : 0.f;
  if (!rates.empty()) {
    std::sort(rates.begin(), rates.end());
    // nearest-rank percentiles
    auto pct = [&](double p) {
      size_t k = (size_t)ceil(p * (double)rates.size());
      if (k < 1) k = 1;
      return (float)rates[k - 1];
    };
    out->acceptance_p50 = pct(0.50);
    out->acceptance_p95 = pct(0.95);
    out->acceptance_p99 = pct(0.99);
    double mean = 0;
    for (double v : rates) mean += v;
    out->acceptance_mean = (float)(mean / rates.size());
  }
  if (steps_total > 0) {
    out->emitted_per_step = (float)(em_total / steps_total);
    out->speculative_efficiency =
        (float)((em_total / steps_total) / (1.0 + (gamma_total / steps_total) * cfg->draft_cost));
  }
  return SPEC_OK;
}

spec_status spec_step_stats(const int32_t* accepted_len, const int32_t* path, const int32_t* parent,
                            int32_t B, int32_t M, spec_step_stats_out* out) {
  if (accepted_len == nullptr || out == nullptr || B < 0 || M < 1 || M > SPEC_STEP_MAX_POS - 1)
    return SPEC_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  double twe = 0;
  int tree_steps = 0;
  for (int b = 0; b < B; ++b) {
    const int a = accepted_len[b];
    if (a < 0) {
      ++out->failed;
      continue;
    }
    ++out->requests;
    out->accepted += a;
    out->emitted += a + 1;
    // where the walk stopped: position a + 1 of the draft (1-based) was
    // rejected, or none was (index M: every draft accepted)
    const int pos = a + 1 < M ? a + 1 : M;
    if (pos < SPEC_STEP_MAX_POS) ++out->rejection_pos[pos];
    if (parent != nullptr && path != nullptr) {
      const int32_t* par = parent + (int64_t)b * M;
      // leaves of the drafted tree, and those below the first accepted node
      bool has_kid[SPEC_STEP_MAX_POS] = {};
      for (int c = 1; c < M; ++c)
        if (par[c] >= 0 && par[c] < M) has_kid[par[c]] = true;
      int leaves = 0, hit = 0;
      const int first = a >= 1 ? path[(int64_t)b * M + 1] : -1;
      for (int c = 1; c < M; ++c) {
        if (has_kid[c]) continue;
        ++leaves;
        if (first < 0) continue;
        int x = c;
        for (int guard = 0; guard < M && x > 0 && x < M; ++guard) {
          if (x == first) {
            ++hit;
            break;
          }
          x = par[x];
        }
      }
      if (leaves > 0) {
        twe += (double)hit / (double)leaves;
        ++tree_steps;
      }
    }
  }
  out->tree_width_effective = tree_steps > 0 ? (float)(twe / tree_steps) : -1.f;
  return SPEC_OK;
}

}  // extern "C"
