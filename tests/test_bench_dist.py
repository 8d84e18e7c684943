"""Multi-rank logic of bench.py on CPU (gloo, world size 2): the step time is
the maximum over ranks and the value aggregates every rank's work; the
reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + 5.0 * rank)
    q.put((rank, ms, bench.job_tflops(1e12, world, ms)))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, val in res:
        assert ms == 15.0                       # slowest rank
        assert abs(val - 2 * 1e12 / 15e-3 / 1e12) < 1e-9


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


class _FakeNvml:
    """Stands in for the driver's NVML library: a counter that advances by
    1500 mJ per read."""

    def __init__(self):
        self.mj = 10_000

    def nvmlDeviceGetHandleByUUID(self, uuid, handle_ref):
        return 0 if uuid.startswith(b"GPU-") else 1

    def nvmlDeviceGetHandleByIndex_v2(self, index, handle_ref):
        return 0

    def nvmlDeviceGetTotalEnergyConsumption(self, handle, energy_ref):
        energy_ref._obj.value = self.mj
        self.mj += 1500
        return 0


def test_energy_meter_and_report():
    import bench
    m = bench.EnergyMeter("GPU-1234", nvml=_FakeNvml())
    a, b = m.read_mj(), m.read_mj()
    rep = bench.energy_report(a, b, 3e12)
    assert rep["joules"] == 1.5 and abs(rep["tflop_per_joule"] - 2.0) < 1e-12
    # an unknown device or an unread counter gives no report, not an error
    assert bench.EnergyMeter("bad", nvml=_FakeNvml()).read_mj() is None
    assert bench.energy_report(None, 5, 1.0) is None and bench.energy_report(5, 5, 1.0) is None


def test_clock_aware_fractions():
    """The bench line's clock-aware denominators: the sustained bf16 GEMM scaled
    from the clock it ran at to the kernel's clock (x2 for FP8), and the
    tensor pipes' issue rate at the kernel's clock."""
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"bf16_sustained": 1700.0, "sustained_mhz": 1400.0}
    r = bench.clock_normalised(2000.0, "fp8", peaks, 152, 2100.0)
    assert abs(r["measured_sustained_at_kernel_clock"]["peak"] - 1700.0 * 2 * 1.5) < 1e-9
    assert abs(r["mma_issue_rate_at_kernel_clock"]["peak"] - 16384 * 152 * 2100e6 / 1e12) < 1e-9
    assert abs(r["mma_issue_rate_at_kernel_clock"]["frac"] * r["mma_issue_rate_at_kernel_clock"]["peak"]
               - 2000.0) < 1e-9
    b = bench.clock_normalised(1000.0, "bf16", peaks, 152, 2100.0)
    assert abs(b["measured_sustained_at_kernel_clock"]["peak"] - 1700.0 * 1.5) < 1e-9
    # no clock sampled: only the kernel clock (None) is reported
    assert bench.clock_normalised(1000.0, "fp8", peaks, 152, None) == {"kernel_sm_mhz": None}
