"""The build's staleness check covers every file the kernels are compiled from (CPU only).

`build.build()` recompiles libgs.so when one of its inputs is newer than the library; a
source file it did not list (a header, or the tile's compute body that step_tma.cuh
includes) would leave a stale library after an edit to it.
"""

import os
import re

from bucketized_guidance_step_gb300 import build


def test_every_included_source_is_a_build_input():
    inputs = {os.path.abspath(f) for f in build._inputs()}
    local = set()
    for name in os.listdir(build.CSRC):
        with open(os.path.join(build.CSRC, name), encoding="utf-8") as f:
            text = f.read()
        for inc in re.findall(r'^\s*#include\s+"([^"]+)"', text, flags=re.M):
            for base in (build.CSRC, build.INCLUDE):
                path = os.path.abspath(os.path.join(base, inc))
                if os.path.exists(path):
                    local.add(path)
    assert os.path.abspath(os.path.join(build.INCLUDE, "gs.h")) in local
    assert os.path.abspath(os.path.join(build.CSRC, "step_tma_compute.inc")) in local
    missing = sorted(p for p in local if p not in inputs)
    assert not missing, missing
