"""Checks of the seeded input generators (CPU only)."""
import json
import os

import numpy as np

from medusa_speculative_decoding_heads_gb300 import configs, synth


def test_philox_known_answers():
    kat = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")))
    for v in kat["vectors"]:
        ctr = np.array([int(x, 16) for x in v["ctr"]], dtype=np.uint32)
        key = [int(x, 16) for x in v["key"]]
        out = synth.philox4x32_10(ctr, key)
        assert [int(x) for x in out] == [int(x, 16) for x in v["out"]]


def test_uniforms_range_and_determinism():
    u1, r1 = synth.uniforms_for_step(3, 4, 5, 3)
    u2, r2 = synth.uniforms_for_step(3, 4, 5, 3)
    assert np.array_equal(u1, u2) and np.array_equal(r1, r2)
    assert u1.dtype == np.float32 and (u1 >= 0).all() and (u1 < 1).all()
    assert abs(float(np.concatenate([u1.ravel(), r1.ravel()]).mean()) - 0.5) < 0.15


def test_lengths_and_capacity():
    L = synth.committed_lengths(0, 1000, 1024, 4096)
    assert L.min() >= 1024 and L.max() <= 4096
    assert synth.cache_capacity(L, 111) % 64 == 0 and synth.cache_capacity(L, 111) >= L.max() + 111


def test_workload_node_counts():
    assert [configs.get(n).N for n in configs.ORDER] == [22, 65, 111, 65, 65]
