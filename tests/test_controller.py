"""The host-side controller and metrics (spec_ctrl_*, spec_step_stats),
through the C ABI, on the CPU.

Pinned against the rules the pages state, with hand-worked numbers:
* page 3, dynamic draft length: the acceptance rate of the last 16 steps
  above 60% gives 8 drafts, 30-60% gives 4, below 30% gives 2; a
  temperature above 0.8 gives 1 at once;
* a request whose speculation does not pay over a full window (tokens
  emitted per step below the step's cost, 1 + gamma * 0.02, page 2 §2.3)
  falls back to plain decoding, as does a request the device failed
  (accepted_len = -1: the capacity fallback of page 3's tree section);
* page 2 §5.1 / page 3 observability: the rejection-position histogram,
  the acceptance-rate histogram and percentiles, the fallback rate, and
  the tree width effective (the share of the tree's paths through the
  first accepted node).
"""
import numpy as np
import pytest

from speculative_decoding_verification_19_gb300.controller import (Controller,
                                                                   default_config, step_stats)


def _run(ctrl, accepted_seq, temperature=None):
    g = None
    for a in accepted_seq:
        g = ctrl.update(np.asarray(a, dtype=np.int32), temperature)
    return g


@pytest.mark.parametrize("rate,gamma_after", [
    (0.875, 8),   # above 60%
    (0.5, 4),     # the middle band
    (0.25, 2),    # below 30%
])
def test_dynamic_gamma_bands(rate, gamma_after):
    # each step accepts the same share of the drafts the controller asked for
    c = Controller(1, gamma0=8, cfg=default_config(min_efficiency=0.0))
    g = np.array([8], np.int32)
    for _ in range(16):
        g = c.update(np.array([int(round(rate * g[0]))], np.int32))
    assert list(g) == [gamma_after]


def test_band_edges():
    # exactly 60% is not above 60%: the middle band; exactly 30% is in it too
    c = Controller(2, gamma0=5, cfg=default_config(min_efficiency=0.0))
    g = _run(c, [[3, 3]] * 1)           # 3/5 = 0.6
    assert g[0] == 4
    c = Controller(1, gamma0=10, cfg=default_config(min_efficiency=0.0, max_gamma=63))
    g = _run(c, [[3]])                  # 3/10 = 0.3
    assert g[0] == 4


def test_hot_temperature_sets_one_draft():
    c = Controller(2, gamma0=4)
    g = c.update(np.array([4, 4], np.int32), np.array([0.9, 0.7], np.float32))
    assert list(g) == [1, 8]


def test_fallback_when_speculation_does_not_pay():
    # every draft rejected for a full window: one token per step against a
    # step cost of 1 + 2 * 0.02: plain decoding from then on
    c = Controller(1, gamma0=2)
    g = _run(c, [[0]] * 15)
    assert g[0] == 2
    g = _run(c, [[0]])
    assert g[0] == 0
    g = _run(c, [[0]] * 3)
    assert g[0] == 0
    m = c.metrics()
    assert m["fallback_rate"] == 1.0


def test_device_failure_falls_back():
    c = Controller(3, gamma0=4)
    g = c.update(np.array([2, -1, 4], np.int32))
    assert g[1] == 0 and g[0] > 0 and g[2] > 0
    m = c.metrics()
    assert abs(m["fallback_rate"] - 1 / 3) < 1e-6


def test_metrics_hand_worked():
    # three requests, 4 steps each at gamma 4 (then gamma moves, so only
    # one step is fed per request here): rates 1/4, 2/4, 4/4
    c = Controller(3, gamma0=4, cfg=default_config(min_efficiency=0.0))
    c.update(np.array([1, 2, 4], np.int32))
    m = c.metrics()
    assert m["requests"] == 3
    hist = m["acceptance_hist"]
    assert hist[2] == 1 and hist[5] == 1 and hist[9] == 1 and sum(hist) == 3
    assert abs(m["acceptance_mean"] - (0.25 + 0.5 + 1.0) / 3) < 1e-6
    assert abs(m["acceptance_p50"] - 0.5) < 1e-6 and abs(m["acceptance_p99"] - 1.0) < 1e-6
    # emitted per step (2 + 3 + 5) / 3, cost 1 + 4 * 0.02
    assert abs(m["emitted_per_step"] - 10 / 3) < 1e-5
    assert abs(m["speculative_efficiency"] - (10 / 3) / 1.08) < 1e-5


def test_step_stats_chain():
    s = step_stats(np.array([0, 1, 4, -1, 4], np.int32),
                   path=np.zeros((5, 5), np.int32))
    assert s["requests"] == 4 and s["failed"] == 1
    assert s["accepted"] == 9 and s["emitted"] == 13
    pos = s["rejection_pos"]
    assert pos[1] == 1 and pos[2] == 1 and pos[5] == 2 and sum(pos) == 4


def test_tree_width_effective():
    # root 0 with children 1 and 2; node 1 with children 3 and 4: leaves
    # 2, 3, 4.  Accepting node 1 first hits the paths to 3 and 4: 2/3;
    # accepting node 2 hits one path: 1/3; accepting nothing: 0
    parent = np.array([[-1, 0, 0, 1, 1]] * 3, np.int32)
    path = np.array([[0, 1, 3, -1, -1], [0, 2, -1, -1, -1], [0, -1, -1, -1, -1]], np.int32)
    s = step_stats(np.array([2, 1, 0], np.int32), path=path, parent=parent)
    assert abs(s["tree_width_effective"] - (2 / 3 + 1 / 3 + 0) / 3) < 1e-6
