"""Host logic of bench.py, without a GPU: the replica timing across ranks (two
gloo processes on the CPU), and the byte accounting behind the roofline
numbers, checked against the library's closed-form kivi_cache_bytes."""
import os
import socket
import sys

import numpy as np
import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, ms, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.reduce_max(ms[rank])
        q.put((rank, slowest, bench.whole_job_value(2e9, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    """Each rank times its own replica; every rank ends with the max, and
    the job value counts all ranks' bytes over that time (weak scaling)."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port, ms = 2, _free_port(), [4.0, 5.0]
    procs = [ctx.Process(target=_replica, args=(r, world, port, ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    assert res[0][2] == pytest.approx(2e9 * 2 / 5e-3 / 1e9)


def test_reduce_max_without_process_group():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.whole_job_value(1e9, 1, 1.0) == pytest.approx(1000.0)


def test_dist_env_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (3, 4, 1)


@pytest.mark.parametrize("name", ["llama2_7b_layer", "prefix_store_int4", "prefix_store_int8",
                                  "mistral_gqa", "tiny"])
def test_step_bytes_match_library_closed_form(kivi_lib, name):
    """The stored-bytes part of the encode accounting equals H x
    kivi_cache_bytes per sequence, for keys and values."""
    from kivi_bit_kv_gb300 import abi
    from kivi_bit_kv_gb300 import workloads as W
    w = W.WORKLOADS[name]
    lens = np.array([w.T - 3 * b for b in range(w.B)])
    ab = bench.call_bytes(w, lens, lens + 1)
    fp16 = sum(w.H * int(n) * w.D * 2 for n in lens)
    for which, key in ((0, "quant_keys"), (1, "quant_values")):
        bits = w.bits_k if which == 0 else w.bits_v
        lib = sum(w.H * abi.kivi_cache_bytes(int(n), w.D, bits, w.G, w.R, which) for n in lens)
        assert ab[key] - fp16 == lib


def test_fp16_equivalent_bytes_per_kind():
    from kivi_bit_kv_gb300 import workloads as W
    w = W.WORKLOADS["llama2_7b_layer"]
    lens = np.full(w.B, w.T)
    kv = 2 * w.B * w.H * w.T * w.D * 2
    assert bench.fp16_equiv_bytes(w, "store", lens, lens) == 2 * kv
    assert bench.fp16_equiv_bytes(w, "decode", lens, lens) == kv + 2 * w.B * w.H * w.D * 2
    assert bench.fp16_equiv_bytes(w, "full", lens, lens) == 3 * kv + 2 * w.B * w.H * w.D * 2


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle) prints one JSON line with
    the keys the benchmark contract asks for, on the host cores."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300, check=True)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1
    assert (line["steps"], line["warmup"]) == (1, 1) and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_0_only():
    from types import SimpleNamespace
    args = SimpleNamespace(workload="tiny", steps=1, warmup=1)
    assert bench.run_reference(args, rank=1, world=2) is None


def test_decode_workloads_rotate_over_twice_the_l2():
    """A decode-only workload whose packed cache would stay in L2 between
    steps is timed over enough cache copies to hold at least 2x the L2."""
    import numpy as np
    from kivi_bit_kv_gb300 import workloads as W
    for name in ("mistral_gqa", "streaming"):
        w = W.WORKLOADS[name]
        lens = W.make_lengths(w).numpy().astype(np.int64)
        per = sum(w.H * (bench.slice_bytes(w, int(n), 0) + bench.slice_bytes(w, int(n), 1)) for n in lens)
        n = bench.cache_copies(w, lens, w.Tmax)
        assert n * per >= 2 * bench.L2_BYTES
        assert (n - 1) * per < 2 * bench.L2_BYTES or n == 1
        note = bench.l2_note(bench.KINDS[name], n, per)
        assert ("rotated" in note) == (n > 1)
    # the GQA cache (136 MB) is about one L2: it needs copies
    w = W.WORKLOADS["mistral_gqa"]
    assert bench.cache_copies(w, W.make_lengths(w).numpy(), w.Tmax) >= 2


def test_timed_region_starts_behind_a_device_busy_wait():
    """queue_ahead issues one device-side busy wait of the requested length
    (in clock cycles at up to 2.07 GHz) through torch.cuda._sleep, and does
    nothing where that call does not exist: with the queue empty at the start
    event, the first call's events would also time the host's launch of it."""
    calls = []

    class _Cuda:
        @staticmethod
        def _sleep(cycles):
            calls.append(cycles)

    class _Torch:
        cuda = _Cuda

    bench.queue_ahead(_Torch, ms=2.0)
    assert calls == [int(2.0 * 2.07e6)]

    class _NoSleep:
        cuda = type("cuda", (), {})

    bench.queue_ahead(_NoSleep)  # no busy wait available: no error
    assert calls == [int(2.0 * 2.07e6)]
