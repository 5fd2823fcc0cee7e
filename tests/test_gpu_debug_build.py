"""The device-check build of the library (-DNVFP4_DEBUG).

Its GEMM kernel checks every shared-memory and TMEM range, TMA coordinate
and alignment before the operation it guards; a failed check records
(device fault, check site) in the error word, skips the operation and ends
the kernel through its abort flag. A child process loads that build
(NVFP4_GGEMM_LIB) and (a) runs problems covering pairs of row tiles,
single row tiles with split accumulators, ragged and empty groups, K % 64
(raw scale rows copied by the scale producer's lanes, in 4-byte pieces and
in 16- and 8-byte row classes, and the re-layout path), atom-layout scales
and the 128-column kernel, which must match the oracle with no check
firing; (b) for each check site, for the kernels of both unit counts and
for raw scale rows loaded by TMA and copied by lanes, forces that check to
fail through the
test-only option debug_check_fail (no invalid operation is issued: the
check's own skip path runs), which must come back as NVFP4_ERR_DEVICE_FAULT
naming that site, after which a good call on the same context matches the
oracle."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def child_result():
    from block_scaled_fp4_grouped_gb300 import build
    path = build.build(debug=True)
    env = dict(os.environ, NVFP4_GGEMM_LIB=path)
    res = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_child.py")], env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    out = json.loads(res.stdout.strip().splitlines()[-1])
    assert out["lib"] == path, "the child loaded another build"
    return out


def test_debug_build_matches_the_oracle_with_no_check_firing(child_result):
    for name, worst in child_result["parity"].items():
        assert worst <= 1.0, (name, worst)


@pytest.mark.parametrize("kind", ["tma", "lanes"])
@pytest.mark.parametrize("units", [1, 2])
@pytest.mark.parametrize("site", range(0x21, 0x27), ids=lambda s: hex(s))
def test_a_failed_check_is_reported_with_its_site(child_result, site, units, kind):
    from block_scaled_fp4_grouped_gb300 import binding as nb
    r = child_result["checks"][f"{kind}/{units}/{hex(site)}"]
    assert r["units"] == units and r["split"] == (1 if units == 1 else 0), r
    assert r["status"] == nb.NVFP4_ERR_DEVICE_FAULT, r
    assert r["word"] & 0xFF == nb.NVFP4_ERR_DEVICE_FAULT, hex(r["word"])
    assert (r["word"] >> 8) & 0xFF == site, hex(r["word"])
    assert r["after"] <= 1.0, "a good call after the failed check"
