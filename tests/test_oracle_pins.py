"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_brute_force_exhaustive_small(orc):
    """Every L, w in [1, S+1] for S up to 12 (the pages' invariants at tiny size)."""
    pins.pin_brute(orc, sizes=range(11, 13), seed=17)


def test_three_pass_empty_remote_set_cancels(orc):
    """When no key is remote, remote(all) and remote(window) are the same set:
    the inclusion-exclusion residue must vanish and the local pass remains."""
    import numpy as np

    r = np.random.default_rng(2)
    S, D = 40, 8
    q, k, v = (r.standard_normal((1, S, 2, D)) for _ in range(3))
    o1, l1 = orc.bifocal_prefill(q, k, v, 4, S + 1, 1e4)
    o3, l3 = orc.bifocal_rows_3pass(q, k, v, np.arange(S), S, 4, S + 1, 1e4)
    assert np.max(np.abs(o1 - o3)) <= 1e-15 * max(1.0, np.max(np.abs(o1))) * 10
    assert np.max(np.abs(l1 - l3)) <= 1e-14


def test_oracle_rejects_bad_arguments(orc):
    import numpy as np

    q = np.zeros((1, 4, 3, 8))
    k = np.zeros((1, 4, 2, 8))
    with pytest.raises(ValueError):  # Hq % Hkv != 0
        orc.bifocal_prefill(q, k, k, 4, 2, 1e4)
    q = np.zeros((1, 4, 2, 8))
    with pytest.raises(ValueError):  # w < 1
        orc.bifocal_prefill(q, k, k, 4, 0, 1e4)
    assert orc.group_factor(0, 4) == -1
