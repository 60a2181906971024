"""Host-side logic of bench.py: the rank reduction over a 2-process gloo group, and the reference arm."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env()[:2] == (world, rank)
        mx = bench.reduce_times([1.0 + rank, 10.0 * (world - rank)], "max")
        sm = bench.reduce_times([1.0 + rank], "sum")
        out.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_reduce_times_over_gloo_world_of_two():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, mx, sm in got:
        assert mx == [2.0, 20.0]
        assert sm == [3.0]


def test_reduce_times_without_a_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_times([3.0, 4.0], "max") == [3.0, 4.0]


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env=env)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


class _FakeNvml:
    """Stands in for the driver's NVML: a scripted sequence of (sm MHz, max MHz, watts, reason bits)."""

    def __init__(self, seq):
        self.seq = list(seq)
        self.i = 0
        self.handles = []

    def handle(self, uuid, pci, index):
        self.handles.append((uuid, pci, index))
        return "h"

    def sample(self, h):
        assert h == "h"
        s = self.seq[min(self.i, len(self.seq) - 1)]
        self.i += 1
        return s


def test_nvml_sampler_summarises_only_samples_inside_a_region():
    sys.path.insert(0, ROOT)
    import bench

    smp = bench.NvmlClockSampler(device=3, period_s=0.001, nvml=_FakeNvml([(2070.0, 2070.0, 500.0, 0x4)]))
    assert smp.error is None
    # samples placed by hand: two inside the region, one before and one after it
    smp.samples = [(0.5, 1000.0, 2070.0, 100.0, 0x8), (1.0, 1800.0, 2070.0, 900.0, 0x4),
                   (1.5, 1900.0, 2070.0, 950.0, 0x0), (2.5, 1200.0, 2070.0, 300.0, 0x40)]
    smp.region("a", 0.9, 2.0)
    s = smp.summary("a")
    assert s["samples"] == 2 and s["sm_mhz"] == 1850.0 and s["sm_min_mhz"] == 1800.0
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 950.0 and s["sm_max_mhz"] == 2070.0
    assert smp.summary("missing")["samples"] == 0 and smp.summary("missing")["sm_mhz"] is None


def test_nvml_sampler_thread_collects_and_decodes_reason_bits():
    sys.path.insert(0, ROOT)
    import time

    import bench

    fake = _FakeNvml([(1500.0, 2070.0, 1400.0, 0x8 | 0x20 | 0x40 | 0x4)])
    smp = bench.NvmlClockSampler(period_s=0.001, nvml=fake)
    t0 = time.time()
    smp.start()
    time.sleep(0.05)
    smp.stop()
    smp.region("r", t0, time.time())
    s = smp.summary("r")
    assert s["samples"] >= 5
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert fake.handles and fake.handles[0][2] == 0


def test_nvml_sampler_without_nvml_reports_the_error():
    sys.path.insert(0, ROOT)
    import bench

    class Broken:
        def handle(self, *a):
            raise OSError("no device")

    smp = bench.NvmlClockSampler(nvml=Broken())
    smp.start()
    smp.stop()
    assert smp.nvml is None and "no device" in smp.error
    assert smp.summary()["samples"] == 0


def test_kernel_source_hash_ignores_comments_but_not_code():
    import bench

    src = 'int a = 1; // note\n/* block\n comment */ const char *s = "// kept"; char c = \'/\';\n'
    code = bench._code_only(src)
    assert code == 'int a = 1; const char *s = "// kept"; char c = \'/\';'
    assert bench._code_only(src.replace("note", "another note")) == code
    assert bench._code_only(src.replace("a = 1", "a = 2")) != code
