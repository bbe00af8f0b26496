"""The committed ncu counter files describe the committed kernels.

`bench.py` turns the per-launch counters of profiles/k_count3m_bao_3pcf.json and
profiles/k_count4_small_parity_4pcf.json into the `roofline` objects of its
line, and drops them (null) when the kernel source hashed at capture time is
not the source in the tree. These tests check, without a GPU, that the files
still match the sources and that their figures agree with one another: the
L1 data-pipe share ncu reported equals the wavefronts per launch over the
launch's duration at one wavefront per SM per cycle, and likewise for issue.
"""
import hashlib
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS = 152                        # GB300
SM_MHZ_MAX = 2070.0              # the capture runs with ncu --clock-control none


def _load(name):
    with open(os.path.join(ROOT, "profiles", name)) as f:
        return json.load(f)


def _sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def test_count3_counters_match_the_kernel_source():
    import bench
    d = _load("k_count3m_bao_3pcf.json")
    assert d["kernel_source_sha256"] == bench.kernel_source_hash()
    assert bench.profiled_counters("bao_3pcf") is not None
    assert bench.profiled_counters("large_3pcf") is None       # another workload's counters are not used


def test_parity_counters_match_the_kernel_source():
    d = _load("k_count4_small_parity_4pcf.json")
    assert d["sources"], "the file names the sources it was hashed over"
    assert d["kernel_source_sha256"] == _sha(d["sources"])


@pytest.mark.parametrize("name, wf, dur, pct", [
    ("k_count3m_bao_3pcf.json", "l1_wavefronts_per_captured_launch", "duration_captured_s", "l1_data_pipe_pct"),
    ("k_count4_small_parity_4pcf.json", "l1_wavefronts_per_launch", "duration_s", "l1_data_pipe_pct"),
])
def test_l1_share_agrees_with_wavefronts_and_duration(name, wf, dur, pct):
    d = _load(name)
    share = d[wf] / (d[dur] * SMS * SM_MHZ_MAX * 1e6)
    # the clock under the capture may sit a little below its maximum
    assert d[pct] / 100 == pytest.approx(share, rel=0.06), (share, d[pct])


@pytest.mark.parametrize("name, inst, dur", [
    ("k_count3m_bao_3pcf.json", "warp_inst_per_captured_launch", "duration_captured_s"),
    ("k_count4_small_parity_4pcf.json", "warp_inst_per_launch", "duration_s"),
])
def test_issue_share_agrees_with_instructions_and_duration(name, inst, dur):
    d = _load(name)
    share = d[inst] / (d[dur] * SMS * 4 * SM_MHZ_MAX * 1e6)    # four schedulers per SM
    assert d["issue_active_pct"] / 100 == pytest.approx(share, rel=0.06), (share, d["issue_active_pct"])


def test_count3_scaling_to_the_full_launch():
    d = _load("k_count3m_bao_3pcf.json")
    # the capture ran the same kernel on a 1/16-scale catalogue; per-edge and
    # per-triangle figures are scaled to one full-size launch
    assert d["scale_to_full"] == pytest.approx(6678002066 / 374084638)
    assert d["dram_bytes_per_full_launch"] == pytest.approx(d["dram_bytes_per_captured_launch"] * d["scale_to_full"])
    tri = 2035238119864 / 112384362712
    assert d["l1_wavefronts_per_full_launch"] == pytest.approx(d["l1_wavefronts_per_captured_launch"] * tri)
    assert d["warp_inst_per_full_launch"] == pytest.approx(d["warp_inst_per_captured_launch"] * tri)
    assert d["shared_atom_lane_ops_per_full_launch"] == 2035238119864    # one add per closed triangle
