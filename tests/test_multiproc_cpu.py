"""The N>1 path of bench.py on CPU: two gloo ranks (127.0.0.1).

The work shards with no data-path exchange (replicas), so the only collective is
the MAX all-reduce of the per-rank time; the whole-job value is N x the units of
one rank over the slowest rank's time.  A rank that fails before the collective
must make the other rank's collective fail (short timeout), not hang."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, out, fail_rank):
    import datetime

    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=10))
    try:
        if rank == fail_rank:
            raise SystemExit(3)  # leaves before the collective, between steps
        ms, value = bench.aggregate_over_ranks(local_ms[rank], 2.0, world, "cpu")
        out.put((rank, ms, value))
    except SystemExit:
        raise
    except Exception as exc:  # the surviving rank sees the collective fail
        out.put((rank, "error", type(exc).__name__))
    finally:
        if rank != fail_rank:
            dist.destroy_process_group()


def _run(local_ms, fail_rank=-1):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, local_ms, q, fail_rank)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    res = {}
    while not q.empty():
        r = q.get()
        res[r[0]] = r[1:]
    return res, [p.exitcode for p in procs]


def test_two_gloo_ranks_take_max_time_and_sum_units():
    res, codes = _run([4.0, 5.0])
    assert codes == [0, 0]
    for r in (0, 1):
        ms, value = res[r]
        assert ms == 5.0
        assert value == pytest.approx(2 * 2.0 / 5e-3)


def test_rank_that_leaves_makes_the_collective_fail_not_hang():
    res, codes = _run([4.0, 5.0], fail_rank=1)
    assert codes[1] == 3
    assert res.get(0, (None,))[0] == "error"


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench

    ms, value = bench.aggregate_over_ranks(8.0, 3.0, 1)
    assert ms == 8.0 and value == pytest.approx(3.0 / 8e-3)


def test_both_arms_name_every_workload_alike():
    """The GPU arm and the oracle (reference) arm take metric, unit and the
    workload part of the config from the same tables, for every workload."""
    import bench
    from cascaded_reductions_pass_gb300 import inputs

    for name, w in inputs.WORKLOADS.items():
        metric, unit, bound = bench.METRICS[w.kind]
        assert unit in ("TFLOP/s", "GB/s") and bound in ("tensor", "hbm")
        assert (unit == "TFLOP/s") == (w.kind == "attn")
        cfg = bench.workload_config(w)
        assert cfg["workload"] == name and cfg["dtype"] == w.dtype and cfg["seed"] == w.seed
        assert all(cfg[k] == v for k, v in w.dims.items())


def test_compact_summary_names_every_workload_within_the_line_tail():
    """The bench line ends with a compact summary of every workload (the five
    configurations first); it must fit in the last ~2 KB of the line."""
    import json

    import bench
    from cascaded_reductions_pass_gb300 import inputs

    def fake(name):
        return {"value": 1234.5678, "unit": "GB/s", "ms_per_step": 0.123456,
                "roofline": {"frac": 0.912345, "bound": "hbm", "traffic": 2168282112},
                "e2e": {"value": 187.654321}}

    names = list(inputs.WORKLOADS)
    head = "attn_fwd_f16_d64"
    parts = {n: fake(n) for n in names if n != head}
    abl = {"layernorm_residual_bf16": {"variants": {str(i): {"slowdown_vs_fused": 1.0 + i} for i in range(4)}},
           "softmax_xent_bf16": {"variants": {str(i): {"slowdown_vs_fused": 1.0 + i} for i in range(3)}}}
    s = bench.compact_summary(head, fake(head), {"value": 500.0}, parts, abl)
    keys = list(s)
    assert keys[:5] == [f"cfg{i + 1} {n}" for i, n in enumerate(bench.CONFIG_ORDER)]
    assert len(keys) == len(names) + 1
    assert len(json.dumps({"summary": s})) < 1900
