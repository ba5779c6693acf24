"""The CPU baseline's sampling (test infrastructure of the benchmark): the single-process and
the all-cores forms time the same count of query-layers, and the all-cores form spreads its
queries over spawned processes."""
from fp4_compressed_sparse_02_gb300 import synth
from oracle import timing


def test_single_and_parallel_samples_count_the_same_layers():
    cfg = dict(synth.DEC128K)
    one = timing.time_sample(4096, 3, cfg)
    many = timing.time_sample_parallel(4096, 3, cfg, 2)
    assert one["query_layers"] == many["query_layers"] == 3 * 20
    assert many["procs"] == 2 and many["seconds"] > 0 and one["seconds"] > 0


def test_layer_steps_walk_the_schedule():
    import numpy as np
    cfg = dict(synth.DEC128K)
    r = np.random.default_rng(0)
    xs = [timing.make_query(r, 4096, cfg)]
    st = timing.LayerSteps(xs, 4096, cfg)
    outs = [st.step() for _ in range(21)]          # a whole query-step, then its first layer again
    assert st.i == 21
    full = timing.run_query(timing.make_query(np.random.default_rng(0), 4096, cfg), 4096, cfg)
    for (o, l), (_, _, ro, rl) in zip(outs[:20], full):
        np.testing.assert_array_equal(o, ro)       # layer by layer = the 20-layer step
        np.testing.assert_array_equal(l, rl)
