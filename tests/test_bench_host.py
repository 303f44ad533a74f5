"""Host helpers of bench.py that need no GPU."""
import numpy as np

import bench


def test_spread_is_p10_median_p90():
    ms = list(np.arange(1.0, 11.0))          # 1..10
    got = bench._spread(ms[::-1])
    assert got == {"p10": 1.9, "median": 5.5, "p90": 9.1}
    assert bench._spread([2.5]) == {"p10": 2.5, "median": 2.5, "p90": 2.5}


def test_split_partition_only_for_two_launches():
    assert bench._split_partition(0, 30000, 1) == 0
    assert bench._split_partition(0, 30000, 2) == 512
    assert bench._split_partition(256, 30000, 2) == 256


def test_packed_step_round_trip():
    """The e2e step's inputs packed into one buffer come back bit for bit,
    each piece 256-byte aligned."""
    import torch
    g = torch.Generator().manual_seed(1)
    ts = {"q": torch.randn(3, 5, 8, generator=g).to(torch.bfloat16),
          "slot_mapping": torch.arange(7, dtype=torch.int64) * 3,
          "block_tables": torch.randint(0, 99, (3, 4), generator=g, dtype=torch.int32),
          "empty": torch.empty(0, 2, dtype=torch.int64),
          "plan": torch.from_numpy(np.arange(11, dtype=np.int32))}
    buf, layout = bench._pack_pinned(ts)
    back = bench._unpack(buf, layout)
    for k, t in ts.items():
        assert layout[k][0] % 256 == 0
        assert back[k].dtype == t.dtype and back[k].shape == t.shape
        assert torch.equal(back[k].view(torch.uint8) if t.numel() else back[k],
                           t.view(torch.uint8) if t.numel() else t)


def test_traffic_only_for_the_kernel_it_was_captured_on():
    """A stored DRAM-traffic ratio scales to the run's bytes only for its own
    workload and kernel, and only while that kernel's sources are unchanged."""
    import json
    import os
    from types import SimpleNamespace
    with open(os.path.join(bench.ROOT, "profiles", "decode_traffic.json")) as f:
        stored = json.load(f)
    for name, per_kernel in stored.items():
        cfg = SimpleNamespace(name=name)
        for k in bench.KERNEL_SOURCES:
            e = per_kernel.get(k)
            fresh = e is not None and e["source_sha"] == bench.kernel_source_sha(k)
            want = int(e["traffic_per_algorithmic_byte"] * 1_000_000) if fresh else None
            assert bench.traffic_for(cfg, k, 1_000_000) == want
        assert set(per_kernel) <= set(bench.KERNEL_SOURCES)
    assert bench.traffic_for(SimpleNamespace(name="no_such_workload"), "pa_decode_kernel", 1) is None
    # every kernel's sources include the headers its file includes
    for k, srcs in bench.KERNEL_SOURCES.items():
        assert len(set(srcs)) == len(srcs)
        assert bench.kernel_source_sha(k) != ""
    assert set(bench.KERNEL_SOURCES["pa_cascade_kernel"]) < set(bench.KERNEL_SOURCES["pa_cascade_tc05_kernel"])


def test_host_step_op_runs_without_a_gpu():
    """bench.py --op host_step times a step's host bookkeeping on the host
    cores alone and prints one JSON line with the pool and planner figures."""
    import json
    import os
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--op", "host_step",
                        "--config", "shared_prefix_bf16", "--steps", "3", "--warmup", "1"],
                       cwd=bench.ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["op"] == "host_step" and line["config"]["workload"] == "shared_prefix_bf16"
    for k in ("pool_append_slots_us", "pool_per_sequence_us", "plan_shared_prefix_us"):
        assert line[k] > 0


def test_staging_packs_a_step_and_views_it_back():
    """The wall-clock loop's per-step staging: tables, lengths, slots, pairs
    and plan packed 256-byte aligned come back bit for bit as typed views."""
    import torch
    rng = np.random.default_rng(3)
    st = bench._Staging(1 << 16, torch.device("cpu"))
    arrays = [("bt", rng.integers(-1, 999, (5, 7)).astype(np.int32)),
              ("cl", rng.integers(0, 99, 5).astype(np.int32)),
              ("slots", rng.integers(0, 1 << 40, 9).astype(np.int64)),
              ("pairs", rng.integers(0, 99, (2, 2)).astype(np.int64)),
              ("plan", np.arange(13, dtype=np.int32))]
    n, views = st.pack(arrays)
    assert n % 256 == 0 and all(o % 256 == 0 for o, *_ in views.values())
    st.dev[:n].copy_(st.host[:n])
    back = st.device_views(views)
    for name, a in arrays:
        assert np.array_equal(back[name].numpy(), a)
