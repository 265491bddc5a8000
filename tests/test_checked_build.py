"""The range-checked build (libmedusa_checked.so) and guard bytes around every buffer.

Each library runs tests/_guarded_step.py in a process of its own (the environment
variable MEDUSA_CHECKED=1 makes the binding load the checked build): small steps
whose outputs, workspace and KV cache sit between guard bytes must match the
oracle with the guards intact and nothing reported; corrupted token ids, paths
and page ids must stay inside their buffers, and only the checked build reports
them (MEDUSA_CHECK_TOKEN, _PATH and _PAGE).
"""
import json
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.gpu
@pytest.mark.parametrize("checked", [False, True])
def test_guarded_steps(checked):
    env = dict(os.environ, MEDUSA_CHECKED="1" if checked else "0")
    r = subprocess.run([sys.executable, os.path.join(HERE, "_guarded_step.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert r.returncode == 0 and lines, f"rc={r.returncode}\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
    out = json.loads(lines[-1])
    assert out["ok"] and out["checked"] == checked
    if checked:
        assert out["codes"]["token"] & 1 and out["codes"]["path"] & 4 and out["codes"]["page"] & 8
    else:
        assert out["codes"] == {"token": 0, "path": 0, "page": 0}


def test_both_builds_export_the_check_entry_points():
    """Both libraries load without a GPU and say which build they are."""
    import ctypes
    sys.path.insert(0, os.path.dirname(HERE))
    from medusa_speculative_decoding_heads_gb300 import _build, binding
    _build.build()
    for path, want in ((binding.LIB_PATH, 0), (binding.LIB_CHECKED_PATH, 1)):
        lib = ctypes.CDLL(path)
        lib.medusa_checked_build.restype = ctypes.c_int
        assert lib.medusa_checked_build() == want
        assert hasattr(lib, "medusa_poll_checks")
