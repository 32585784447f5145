"""The bench's buffer-set rule: the sets a timed loop rotates through hold at least three
times L2 together, so no call finds its inputs in L2 (no flush is used), and a workload
whose one set exceeds L2 uses two sets."""
import bench
import workloads as W

L2 = 126 * 2**20  # the GB300's L2 (the bench reads the real size from the device)


def _per_set(name):
    w = W.WORKLOADS[name]
    return (W.compulsory_bytes(w.op, "forward", w.N, w.D)
            + W.compulsory_bytes(w.op, "backward", w.N, w.D))


def test_large_workloads_use_two_sets():
    for name in ("add_rmsnorm_32768x4096", "rmsnorm_16384x4096", "layernorm_2048x16384",
                 "rmsnorm_4096x32768", "layernorm_1024x131072"):
        assert _per_set(name) > L2, name
        assert bench.n_buffer_sets(name, L2) == 2, name


def test_small_workloads_rotate_through_three_times_l2():
    for name in W.WORKLOAD_ORDER:
        n = bench.n_buffer_sets(name, L2)
        assert n >= 2
        assert n * _per_set(name) >= 3 * L2 or n == 4096, name


def test_config_states_the_rule():
    c = bench.bench_config(bench.DEFAULT_WORKLOAD, 1)
    assert c["l2"].startswith("not flushed") and "more than L2" in c["l2"]
