"""The benchmark's accounting on the CPU: the algorithmic bytes and FLOPs its roofline divides
by, and the rule that reports ncu traffic only for the kernel source it was captured from."""
import hashlib
import os

import bench
from synth import workload as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_layer_bytes_closed_form():
    # one token, E=288, k=8, H=3072, I=1024, no shared expert, 8 experts touched: per expert
    # 3*H*I elements (W13 is 2I x H, W2 is H x I) at 4 bits + one E4M3 byte per 16, and two
    # fp32 tensor scales; x in and y out in bf16; the fp32 logits
    H, I, E = 3072, 1024, 288
    per_expert = 3 * H * I // 2 + 3 * H * I // 16 + 8
    expect = 8 * per_expert + 2 * H * 2 + E * 4
    assert expect == 42480832
    assert bench.layer_bytes(wl.DECODE_B1_E288, 8) == expect


def test_layer_bytes_shared_expert_and_tokens():
    spec = wl.DECODE_B1_E512          # T=1, E=512, k=10, H=4096, I=1024, shared expert
    H, I, E, T = spec.H, spec.I, spec.E, spec.T
    per_expert = 3 * H * I // 2 + 3 * H * I // 16 + 8
    # the shared expert streams like one more expert, plus its bf16 gate vector
    assert bench.layer_bytes(spec, 10) == 11 * per_expert + T * H * 4 + T * E * 4 + H * 2


def test_layer_flops():
    spec = wl.PREFILL_T2048
    pairs = spec.T * spec.k
    # 2 FLOP per multiply-add over the gate, up and down products of every (token, expert) pair
    assert bench.layer_flops(spec, pairs) == 2.0 * pairs * (2 * spec.I * spec.H + spec.H * spec.I)


def _table_rows():
    rows = {}
    for line in open(os.path.join(ROOT, "profiles", "dram_traffic.md")):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[3].isdigit():
            rows[cells[0]] = (cells[1], cells[2], int(cells[3]))
    return rows


def test_measured_traffic_follows_the_source_hash():
    rows = _table_rows()
    assert wl.DECODE_B1_E288.name in rows          # the default workload has a capture row
    for name, (src, sha, nbytes) in rows.items():
        path = os.path.join(ROOT, "nvfp4_mixture_experts_02_gb300", "csrc", src)
        cur = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
        assert bench.measured_traffic(name) == (nbytes if cur == sha else None), name
    assert bench.measured_traffic("no_such_workload") is None


def test_measured_traffic_is_dropped_when_the_source_changes(tmp_path, monkeypatch):
    # a copy of the tree's layout whose kernel source no longer matches the table
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "nvfp4_mixture_experts_02_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("// v2\n")
    sha_v1 = hashlib.sha256(b"// v1\n").hexdigest()[:16]
    sha_v2 = hashlib.sha256(b"// v2\n").hexdigest()[:16]
    table = tmp_path / "profiles" / "dram_traffic.md"
    table.write_text(f"| w1 | k.cu | {sha_v1} | 100 | c |\n| w2 | k.cu | {sha_v2} | 200 | c |\n")
    monkeypatch.setattr(bench.os.path, "abspath",
                        lambda p, _real=os.path.abspath: str(tmp_path / "bench.py")
                        if p == bench.__file__ else _real(p))
    assert bench.measured_traffic("w1") is None
    assert bench.measured_traffic("w2") == 200



def test_clock_summary_keeps_the_timed_window():
    clk = bench.ClockSampler(0)
    row = "0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    clk.lines = [(1.0, row.format(sm=1000, cap="Not Active")),      # before: idle clock
                 (2.0, row.format(sm=2070, cap="Active")),
                 (2.1, row.format(sm=2060, cap="Not Active")),
                 (9.0, row.format(sm=800, cap="Not Active"))]        # after
    clk.t_start, clk.t_end = 1.9, 2.2
    s = clk.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2065 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region and kernel replays"
    clk.t_start, clk.t_end = 5.0, 5.1                                # no sample inside
    s = clk.summary()
    assert s["samples"] == 4 and s["window"].startswith("warm-up")


def test_gpus_must_match_the_launched_world(tmp_path):
    import subprocess
    import sys
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and "WORLD_SIZE" in r.stderr
