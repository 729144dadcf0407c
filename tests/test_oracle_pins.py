"""The float64 CPU oracle against what the pages and the mathematics fix
(printed probabilities, hand-derived cases, closed forms, scipy, finite
differences).  CPU only."""
import pytest

import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_CHEAP, ids=lambda f: f.__name__)
def test_pin(oracle_mod, pin):
    pin(oracle_mod)


def test_printed_probabilities():
    pins.pin_printed_probabilities()


def test_advantage_monte_carlo(oracle_mod):
    pins.pin_advantage_monte_carlo(oracle_mod)


def test_thread_count_does_not_change_results(oracle_mod):
    import numpy as np
    from vocab_wide_logprob_gb300 import workloads as wl
    w = wl.TINY
    ids = wl.make_ids(w)
    z, dt = wl.logits_as_numpy(wl.make_logits_cpu(w))
    _, lens = oracle_mod.mask(ids, w.P, w.C, w.eos_id)
    n0 = oracle_mod.threads()
    try:
        oracle_mod.set_threads(1)
        a = oracle_mod.logp(z, dt, w.P, w.C, ids, lens)
        oracle_mod.set_threads(5)
        b = oracle_mod.logp(z, dt, w.P, w.C, ids, lens)
    finally:
        oracle_mod.set_threads(0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert n0 >= 1
