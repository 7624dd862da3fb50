"""Host-side checks of the benchmark's workload description: the packed expert bytes it reports
(the `l2` field of the JSON line's config) against the bytes the generator actually produces."""
import dataclasses
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
import harness as H  # noqa: E402


def test_qmat_bytes_glm_shapes():
    # int4-g128 [2048][7168]: 7,340,032 B codes + 56 groups x 2 B scales + 28 B zero nibbles per row
    assert bench.qmat_bytes(H.Q_INT4_G128, 2048, 7168) == 7_340_032 + 229_376 + 57_344
    # int8 per channel: codes + fp32 scale + uint8 zero point per row
    assert bench.qmat_bytes(H.Q_INT8_PC, 2048, 7168) == 2048 * 7168 + 2048 * 5
    # one GLM-class int4 expert (gate, up, down)
    per = 2 * bench.qmat_bytes(H.Q_INT4_G128, 2048, 7168) + bench.qmat_bytes(H.Q_INT4_G128, 7168, 2048)
    assert per == 22_880_256


@pytest.mark.parametrize("name", ["tiny", "decode", "mtp_verify", "prefill", "stacked"])
def test_expert_set_bytes_match_generated(name):
    w = H.WORKLOADS[name]
    # reduced shapes with the workload's quantisation types and shared-expert presence;
    # K = 384 gives an odd number of int4 groups per row (zero-point nibbles padded to a byte)
    small = dataclasses.replace(w, d=384, F=256, E=3, F_shared=128 if w.F_shared else 0)
    total = 0
    for l in range(small.n_layers):
        layer = small.layer(l)
        banks = [layer.experts] + ([layer.shared] if layer.shared is not None else [])
        for b in banks:
            total += b.gate.nbytes + b.up.nbytes + b.down.nbytes
    assert bench.expert_set_bytes(small) == total


def test_config_names_the_workload_only():
    w = H.WORKLOADS["decode"]
    c = bench.workload_config(w, 1, 1)
    assert c["workload"].startswith("decode:") and "T=1" in c["workload"]
    assert "host_generation_s" not in c
    assert "5.86 GB" in c["l2"]
