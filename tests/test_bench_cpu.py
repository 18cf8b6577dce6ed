"""bench.py's host-side harness without a GPU: the oracle timed on every host
core (one spawned process per core over row slices in shared memory) counts
the work it was given and reports the cores it used."""
import numpy as np

import bench


def test_oracle_on_every_core_counts_its_work(oracle_mod):
    K = bench.K
    a = np.zeros((6, K), dtype=np.uint16)
    b_cm = np.zeros((40, K), dtype=np.uint16)
    bias = np.zeros(40, dtype=np.float32)
    pool = bench.OracleCores(a, b_cm, bias, max_rows=6)
    try:
        assert pool.cores == bench._host_cores() >= 1
        t, flops = pool.run(6, 40)
        assert t > 0 and flops == 2.0 * 6 * 40 * K
        t, flops = pool.run(100, 8)          # rows beyond the shared sample are cut
        assert flops == 2.0 * 6 * 8 * K
    finally:
        pool.close()


def test_sample_rows_scale_with_cores():
    per_out = 1e-4                           # seconds per output on one core
    r1 = bench._rows_for(10.0, per_out, 1)
    r16 = bench._rows_for(10.0, per_out, 16)
    assert r16 >= 15 * r1 and r1 >= 1
