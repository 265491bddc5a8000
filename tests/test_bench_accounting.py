"""The benchmark's byte accounting (roofline numerator) against hand counts of each workload.

Hand counts at the mean committed length, nothing accepted (acc = 0), in GB (1e9 bytes):
  7B  B=1:  heads 4(4096^2 + 4096*32000)*2 + 4096*2 = 1182.81 MB; KV 2048*32*128*2*2 = 33.55 MB;
            tree Q/K/V 65*96*128*2 = 1.60 MB; O 0.53 MB; target row 64 KB          -> 1.2186
  13B B=8:  heads 5(5120^2 + 5120*32000)*2 + 8*5120*2 = 1900.50 MB; logits 2*8*5*32000*4 = 10.24 MB;
            KV 8*2560*40*128*4 = 419.43 MB; tree 27.28 MB; O 9.09 MB; rows 0.51 MB  -> 2.3672
  33B B=16: heads 4(6656^2 + 6656*32000)*2 + 16*6656*2 = 2058.22 MB; KV 16*8192*52*128*4 = 3489.66 MB;
            tree 33.23 MB; O 11.08 MB; rows 1.02 MB                                -> 5.6046
  GQA B=32: heads 1182.93 MB; logits 32.77 MB; KV 32*10240*8*128*4 = 1342.18 MB; tree 25.56 MB;
            O 17.04 MB; rows 2.05 MB                                               -> 2.6026
"""
import numpy as np
import pytest

import bench
from medusa_speculative_decoding_heads_gb300 import configs


@pytest.mark.parametrize("name,gb", [("vicuna7b_b1", 1.2186), ("vicuna13b_b8", 2.3672), ("vicuna33b_b16", 5.6046),
                                     ("gqa7b_b32", 2.6026)])
def test_step_bytes_match_hand_counts(name, gb):
    w = configs.get(name)
    L = np.full(w.B, int(np.mean(w.L_range)))
    by = bench.algorithmic_bytes(w, L, np.zeros(w.B, dtype=np.int64), w.modes[0])
    assert abs(by["total"] / 1e9 - gb) < 5e-5 * gb + 1e-4
    assert by["total"] == sum(v for k, v in by.items() if k != "total")


def test_shared_projection_is_counted_once():
    w, s = configs.get("vicuna7b_b1"), configs.get("vicuna7b_b1_shared")
    L, acc = np.array([2048]), np.array([0])
    a = bench.algorithmic_bytes(w, L, acc, w.modes[0])["heads"]
    b = bench.algorithmic_bytes(s, L, acc, s.modes[0])["heads"]
    assert a - b == (w.K - 1) * w.d * w.V * 2   # three of the four vocab matrices are not streamed
