"""The workload registry: names, overrides as bench.py's sweeps use them, and a calibrated Delta
for every workload (host logic only; no GPU)."""
import json
import os

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "delta_calibration.json")


def test_registry_names():
    for name, spec in synth.WORKLOADS.items():
        assert spec.name == name
        assert synth.spec_for(name) is spec


def test_overrides_replace_fields_including_the_name():
    spec = synth.spec_for("128k_gqa_student_t", lengths=(4096,), name="structure_4k")
    base = synth.spec_for("128k_gqa_student_t")
    assert spec.name == "structure_4k" and spec.lengths == (4096,)
    assert (spec.seed, spec.key_dist, spec.num_q_heads) == (base.seed, base.key_dist, base.num_q_heads)
    assert base.lengths == (131072,)   # the registry entry itself is unchanged


def test_every_workload_has_a_calibrated_delta():
    cal = json.load(open(GOLDEN))["workloads"]
    assert set(cal) == set(synth.WORKLOADS)
    for name, entry in cal.items():
        assert entry["delta"] > 0, name
        assert entry["delta"] < min(synth.WORKLOADS[name].lengths), name
