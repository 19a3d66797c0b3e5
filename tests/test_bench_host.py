"""Host-side arithmetic of bench.py (no GPU): algorithmic bytes, the
roofline fields, the launch count per call and the guard that drops a
recorded DRAM traffic figure once the kernel sources change."""
import json
import os

import pytest

import bench
import gdn_inputs


def test_prefill_alg_bytes_t4096():
    w = gdn_inputs.WORKLOADS["prefill_t4096"]
    tok = 1 * 4096
    qk = tok * 16 * 128 * 2 * 2          # q and k, bf16
    vy = tok * 32 * 128 * 2 * 2          # v and y, bf16
    gb = tok * 32 * 2 * 2                # g and beta, bf16
    state = 2 * 1 * 32 * 128 * 128 * 4   # state in and out, fp32
    assert bench.prefill_alg_bytes(w) == qk + vy + gb + state == 105381888


def test_decode_alg_bytes_b64():
    w = gdn_inputs.WORKLOADS["decode_b64"]
    state = 2 * 64 * 32 * 128 * 128 * 4
    assert bench.decode_alg_bytes(w) == state + 64 * 16 * 128 * 2 * 2 + 64 * 32 * 128 * 2 * 2 \
        + 64 * 32 * 2 * 2


def test_roofline_fields():
    r = bench.roofline(105381888, 123.5e-6, 6781.4, "measured", traffic=152.0e6)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6781.4
    assert r["achieved"] == pytest.approx(105381888 / 123.5e-6 / 1e9, abs=0.05)
    assert r["frac"] == pytest.approx(r["achieved"] / 6781.4, abs=1e-4)
    assert r["traffic"] == 152000000
    assert bench.roofline(1, 1.0, 1.0, "fallback")["traffic"] is None


class _Props:
    multi_processor_count = 152


@pytest.mark.parametrize("name,expect", [
    ("prefill_t4096", 1),       # fused cooperative kernel: 3 * 32 <= 152
    ("prefill_t4096_f16", 1),
    ("prefill_t65536", 1),
    ("prefill_b4_t2048", 2),    # 3 * 192 > 152: prep then scan
    ("prefill_b64_t16", 1),     # T <= 32: the short-T kernel
    ("fp32_t64", 2),            # fp32 chunked path: intra-chunk then scan
])
def test_prefill_launch_count(monkeypatch, name, expect):
    monkeypatch.setattr(bench.torch.cuda, "get_device_properties", lambda dev: _Props())
    assert bench.prefill_launches(gdn_inputs.WORKLOADS[name], None) == expect


def test_traffic_guard_follows_the_sources(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1")
    import hashlib
    sha = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    monkeypatch.setattr(bench, "_KDIR", str(tmp_path))
    monkeypatch.setitem(bench.MEASURED_TRAFFIC, "probe", {"sources": ["k.cu"], "sha": sha,
                                                         "bytes": 1.0e6})
    assert bench.measured_traffic("probe") == 1.0e6
    src.write_bytes(b"kernel v2")
    assert bench.measured_traffic("probe") is None


def test_recorded_traffic_entries_are_well_formed():
    """Every recorded DRAM traffic figure belongs to a workload of the plan and
    names kernel sources that exist (its hash then decides whether the line
    reports it or null)."""
    for key, entry in bench.MEASURED_TRAFFIC.items():
        assert key in gdn_inputs.WORKLOADS, key
        assert entry["bytes"] > 0 and len(entry["sha"]) == 16
        for name in entry["sources"]:
            assert os.path.exists(os.path.join(bench._KDIR, name)), name


def test_reference_arm_config_matches_ours():
    """Both arms print the same ``config`` object for the same workload."""
    w = gdn_inputs.WORKLOADS["prefill_t4096"]
    assert bench.workload_config(w, 1) == bench.workload_config(w, 1)
    c = bench.workload_config(w, 2)
    assert c["workload"] == "prefill_t4096" and c["parallelism"] == "replicas x2"
    for name in bench.EXTRA_PREFILL:
        assert name in gdn_inputs.WORKLOADS


def test_measured_peaks_file_is_used_when_present():
    hbm, tf, kind = bench.load_peaks()
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        assert kind == "measured" and hbm == float(p["hbm_gbs"])
    else:
        assert kind == "fallback"
