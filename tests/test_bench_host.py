"""Host-side pieces of the bench (CPU): the clock sampler's parsing of
nvidia-smi samples, the recorded-traffic lookup that is tied to the decode
kernel's sources, the algorithmic byte counts, the whole-job rate, the
timed-region segments of the spread and the CPU model string."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeProc:
    """Stands in for the nvidia-smi process the sampler stops."""

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_parses_samples(tmp_path):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    with open(cs.path, "w") as f:
        f.write("2070, 2070, 800.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
        f.write("2055, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")
        f.write("not a sample\n")
        f.write("[N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    cs.proc, cs.fh = _FakeProc(), open(os.devnull, "w")
    r = cs.stop()
    assert r == {"sm_mhz": 2062.5, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2}
    assert not os.path.exists(cs.path)


def test_clock_sampler_without_nvidia_smi():
    cs = bench.ClockSampler(0)
    assert cs.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_recorded_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    rec = tmp_path / "traffic.md"
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(rec))
    assert bench.recorded_traffic() is None                       # no record
    rec.write_text(f"traffic_bytes_per_launch: 123456\nkernel_source_digest: {bench.decode_kernel_digest()}\n")
    assert bench.recorded_traffic() == 123456
    rec.write_text("traffic_bytes_per_launch: 123456\nkernel_source_digest: 0000000000000000\n")
    assert bench.recorded_traffic() is None                       # sources changed since the capture


def test_committed_traffic_record_is_well_formed():
    """The committed record parses (its digest may lag the sources between a
    kernel change and the next capture; then the bench reports null)."""
    path = os.path.join(ROOT, "profiles", "decode_gemm_qkv_10240x5120.md")
    fields = {}
    for line in open(path):
        if ":" in line and line.split(":", 1)[0] in ("traffic_bytes_per_launch", "kernel_source_digest"):
            k, v = line.split(":", 1)
            fields[k] = v.strip()
    assert int(fields["traffic_bytes_per_launch"]) > 52_000_000
    assert len(fields["kernel_source_digest"]) == 16


def test_algorithmic_bytes():
    # QKV at M = 1: weights + tokens + bf16 output + per-channel scales + the scalar scale
    assert bench.gemm_bytes(1) == 10240 * 5120 + 5120 + 2 * 10240 + 4 * 10240 + 4
    assert bench.norm_bytes(1) == 2 * 5120 + 2 * 5120 + 5120 + 4
    assert bench.step_bytes() == sum(bench.gemm_bytes(m) + bench.norm_bytes(m) for m in (1, 2, 4, 8, 16, 32))
    assert bench.step_bytes() == 317_460_528


def test_whole_job_rate_sums_the_replicas():
    one = bench.whole_job_tbps(1, 317_460_528, 0.11)
    assert abs(one - 317_460_528 / 0.11e-3 / 1e12) < 1e-12
    assert abs(bench.whole_job_tbps(4, 317_460_528, 0.11) - 4 * one) < 1e-12


def test_segment_bounds_split_the_replays_evenly():
    for reps in (1, 2, 5, 7, 10, 103):
        for segments in (1, 3, 5, 8):
            b = bench.segment_bounds(reps, segments)
            assert b[0] == 0 and b[-1] == reps
            lengths = [b[i + 1] - b[i] for i in range(len(b) - 1)]
            assert len(lengths) == min(segments, reps)
            assert min(lengths) >= 1 and max(lengths) - min(lengths) <= 1
    assert bench.segment_bounds(4, 0) == [0, 4]


def test_cpu_model_names_arm_and_x86_parts(tmp_path):
    arm = tmp_path / "arm"
    arm.write_text("processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\n"
                   "CPU part\t: 0xd4f\n\nprocessor\t: 1\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n")
    assert bench.cpu_model(str(arm)).startswith("Neoverse V2 (implementer 0x41 part 0xd4f) (")
    other = tmp_path / "other"
    other.write_text("processor\t: 0\nCPU implementer\t: 0x4e\nCPU part\t: 0x004\n")
    assert bench.cpu_model(str(other)).startswith("(implementer 0x4e part 0x004) (")
    x86 = tmp_path / "x86"
    x86.write_text("processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Example CPU @ 2.00GHz\n")
    assert bench.cpu_model(str(x86)).startswith("Example CPU @ 2.00GHz (")
    assert "logical CPUs)" in bench.cpu_model(str(tmp_path / "missing"))
