"""The benchmark's CPU-baseline runners: every unit of a workload is run once per pass,
in-process and over spawned workers, through the oracle functions as they stand."""
import numpy as np
import pytest

import oracle
from oracle import timing
from paged_kv_attention_28_gb300 import workloads


def _small_decode():
    return workloads.make_paged_decode(7, 3, 4, 2, 16, page_size=16, kv_lens=[40, 17, 64], num_pages=16,
                                       dtype="f32", name="timing_small")


def _small_cascade():
    return workloads.make_cascade(8, 3, 32, (5, 20), 4, 2, 16, page_size=16, num_pages=16,
                                  max_suffix_blocks=2, dtype="f32", name="timing_cascade")


@pytest.mark.parametrize("workers", [1, 2])
def test_decode_runner_runs_every_unit(workers):
    c = _small_decode()
    r = timing.decode_runner(c.q.double().numpy(), c.k_pages.float().numpy(), c.v_pages.float().numpy(),
                             c.block_table.numpy(), c.kv_lens.numpy(), c.scale, workers)
    try:
        assert r.one_pass() == c.batch * c.n_kv_heads
        passes, el = timing.time_passes(r, 0.0)
        assert passes == 1 and el > 0
    finally:
        r.close()


@pytest.mark.parametrize("workers", [1, 2])
def test_cascade_runner_runs_every_request(workers):
    c = _small_cascade()
    r = timing.cascade_runner(c.q.double().numpy(), c.k_pages.float().numpy(), c.v_pages.float().numpy(),
                              c.prefix_table.numpy(), c.prefix_len, c.suffix_table.numpy(),
                              c.suffix_lens.numpy(), c.scale, workers)
    try:
        assert r.one_pass() == c.n_requests
    finally:
        r.close()


def test_cascade_runner_unit_is_the_oracle_on_one_request():
    # the unit function's call on request r gives the whole-batch oracle's rows of r
    c = _small_cascade()
    args = (c.q.double().numpy(), c.k_pages.float().numpy(), c.v_pages.float().numpy(), c.prefix_table.numpy(),
            c.prefix_len, c.suffix_table.numpy(), c.suffix_lens.numpy(), c.scale)
    full_o, full_l = oracle.cascade_decode(*args)
    for r in range(c.n_requests):
        o, l = oracle.cascade_decode(args[0][r:r + 1], args[1], args[2], args[3], args[4], args[5][r:r + 1],
                                     args[6][r:r + 1], args[7])
        np.testing.assert_array_equal(o[0], full_o[r])
        np.testing.assert_array_equal(l[0], full_l[r])
