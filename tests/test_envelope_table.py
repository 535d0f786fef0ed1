"""The oracle's envelope tables (tests/golden/envelope_table_*.txt, written by
make_envelope_table.py from the oracle alone) are present and well formed, and the
end-to-end bound selection of test_gpu_end_to_end_bounds.py picks at least one depth (CPU)."""
import numpy as np

from test_gpu_end_to_end_bounds import BOUNDS, envelope_table, resolvable_depths


def test_tables_cover_every_depth_and_grow_with_it():
    for name in BOUNDS:
        table = envelope_table(name)
        env = {(L, S): e for L, S, e in table}
        assert sorted(env) == sorted((L, S) for L in (1, 2, 6, 18) for S in (1, 2, 10))
        assert all(np.isfinite(e) and e > 0 for e in env.values())
        # one layer-step spreads far less than the whole 18 x 10 decision
        assert env[(18, 10)] > 5 * env[(1, 1)]


def test_bound_selection_is_not_empty():
    for name in BOUNDS:
        depths = resolvable_depths(name)
        assert depths and all(L * S <= 18 * 10 for L, S in depths)
