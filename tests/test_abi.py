"""The C-ABI library loads and exports every entry point include/gs.h declares (CPU only).

Argument checks that return before any CUDA call are exercised here too: they
must answer GS_ERR_INVALID_ARG without a GPU.
"""

import ctypes
import os
import re

import pytest

from bucketized_guidance_step_gb300 import build, gs

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gs.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gs.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:gs_status|const char\*|int32_t)\s+(gs_\w+)\s*\(",
                                 text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(gs.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_abi_version_and_status_strings(lib):
    assert lib.gs_abi_version() == gs.GS_ABI_VERSION
    for code in range(9):
        assert gs.status_string(code) not in ("", "unknown status")
    assert gs.status_string(99) == "unknown status"
    assert gs.status_from_word(0) == gs.GS_OK
    assert gs.status_from_word(gs.GS_DEV_STEP_RANGE) == gs.GS_ERR_STEP_RANGE
    assert gs.status_from_word(gs.GS_DEV_NEED_UNCOND) == gs.GS_ERR_NEED_UNCOND
    assert gs.status_from_word(gs.GS_DEV_SIGMA) == gs.GS_ERR_SIGMA


def _valid_args():
    a = gs.StepArgs()
    a.B, a.C, a.H, a.W, a.dtype = 2, 4, 8, 8, gs.GS_DTYPE_BF16
    a.x = a.x_out = a.uncond = a.cond = 0x1000
    a.sigmas, a.n_sigmas, a.step = 0x2000, 5, 0
    return a


@pytest.mark.parametrize("field,value", [
    ("B", 0), ("C", 0), ("H", -1), ("dtype", 7), ("x", 0), ("x_out", 0), ("sigmas", 0),
    ("n_sigmas", 1), ("step", 4), ("step", -1), ("n_regions", 17), ("n_regions", -1),
])
def test_step_rejects_invalid_arguments(lib, field, value):
    a = _valid_args()
    setattr(a, field, value)
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG


def test_step_rejects_bad_regions_and_missing_branches(lib):
    a = _valid_args()
    a.cond = 0
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG  # no positive branch
    a = _valid_args()
    a.inpaint_mask = 0x3000                                              # mask without original
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    bad = [gs.RegionDesc(0, 0, 9, 4, 1.0, 0, None, 0, 0x4000, 4),     # taller than the frame
           gs.RegionDesc(2, 6, 2, 3, 1.0, 0, None, 0, 0x4000, 4),     # past the right edge
           gs.RegionDesc(0, 0, 2, 4, 1.0, 0, None, 0, 0x4000, 3),     # pitch < w
           gs.RegionDesc(0, 0, 2, 4, 1.0, 0, None, 0, None, 4),       # no output
           gs.RegionDesc(0, 0, 2, 4, -1.0, 0, None, 0, 0x4000, 4),    # negative strength
           gs.RegionDesc(0, 0, 2, 4, 1.0, -2, None, 0, 0x4000, 4)]    # negative feather
    for r in bad:
        a = _valid_args()
        arr = (gs.RegionDesc * 1)(r)
        a.n_regions = 1
        a.regions = ctypes.cast(arr, ctypes.POINTER(gs.RegionDesc))
        assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    a = _valid_args()
    a.n_regions = 1                                                      # regions pointer NULL
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_guided_step(None, None) == gs.GS_ERR_INVALID_ARG


def test_mask_prepare_rejects_invalid_arguments(lib):
    assert lib.gs_mask_prepare(None, 1, 8, 8, 0x1000, 4, 4, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_mask_prepare(0x1000, 0, 8, 8, 0x2000, 4, 4, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_mask_prepare(0x1000, 1, 8, 8, 0x2000, 0, 4, None) == gs.GS_ERR_INVALID_ARG


def test_host_entry_points_reject_invalid_arguments(lib):
    for kw in ({"steps": 0}, {"denoise": 0.0}, {"sigma_min": 0.0}, {"rho": 0.0},
               {"sigma_max": 0.01}):
        args = {"steps": 10}
        args.update(kw)
        steps = args.pop("steps")
        with pytest.raises(gs.GSError):
            gs.sigmas("karras", steps, **args)
    with pytest.raises(gs.GSError):
        gs.sigmas("cosine", 10)
    with pytest.raises(gs.GSError):
        gs.bucket_plan(0, 4)
    with pytest.raises(gs.GSError):
        gs.bucket_plan(10, 0)
    with pytest.raises(gs.GSError):
        gs.bucket_plan(10, 4, curve="table")
    # capacity: a too-small buffer reports the needed length
    d = gs.ScheduleDesc(gs.GS_SCHED_KARRAS, 10, 0.03, 14.6, 7.0, 1.0, -1, -1, 0, 1000,
                        0.00085, 0.012)
    n = ctypes.c_int32(0)
    buf = (ctypes.c_float * 4)()
    assert lib.gs_sigmas(ctypes.byref(d), buf, 4, ctypes.byref(n), None) == gs.GS_ERR_CAPACITY
    assert n.value == 11


def test_step_rejects_invalid_sampler_arguments(lib):
    a = _valid_args()
    a.sampler = 2                                                        # unknown sampler
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    a = _valid_args()
    a.sampler = gs.SAMPLERS["euler_ancestral"]                           # ancestral, no noise
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    a = _valid_args()
    a.model_in_out = 0x5000                                              # model input, no mask
    a.orig_noise = 0x6000
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    a = _valid_args()
    a.inpaint_mask, a.original, a.model_in_out = 0x3000, 0x4000, 0x5000  # ... no orig_noise
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    a = _valid_args()                                                    # model input on x_out
    a.inpaint_mask, a.original, a.orig_noise = 0x3000, 0x4000, 0x6000
    a.model_in_out = a.x_out
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG


_LAYOUT_PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "gs.h"
#define F(S, m) printf(#S " " #m " %zu\n", offsetof(S, m));
int main(void) {
    printf("gs_step_args sizeof %zu\n", sizeof(gs_step_args));
    printf("gs_region sizeof %zu\n", sizeof(gs_region));
    printf("gs_curve_desc sizeof %zu\n", sizeof(gs_curve_desc));
    printf("gs_schedule_desc sizeof %zu\n", sizeof(gs_schedule_desc));
    printf("gs_area sizeof %zu\n", sizeof(gs_area));
    printf("gs_rect sizeof %zu\n", sizeof(gs_rect));
    printf("gs_cond_entry sizeof %zu\n", sizeof(gs_cond_entry));
    printf("gs_cond_chunk sizeof %zu\n", sizeof(gs_cond_chunk));
    printf("gs_step_plan sizeof %zu\n", sizeof(gs_step_plan));
    %FIELDS%
    return 0;
}
"""


def test_ctypes_structs_match_the_header_layout(repo_tmp):
    """Every ctypes mirror in the binding has the C compiler's offsets and size."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pairs = {"gs_step_args": gs.StepArgs, "gs_region": gs.RegionDesc,
             "gs_curve_desc": gs.CurveDesc, "gs_schedule_desc": gs.ScheduleDesc,
             "gs_area": gs.Area, "gs_rect": gs.Rect, "gs_cond_entry": gs.CondEntry,
             "gs_cond_chunk": gs.CondChunk, "gs_step_plan": gs.StepPlan}
    fields = "\n    ".join(f"F({c}, {f})" for c, py in pairs.items() for f, _ in py._fields_)
    src = repo_tmp / "layout.c"
    src.write_text(_LAYOUT_PROBE.replace("%FIELDS%", fields))
    exe = repo_tmp / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True,
                               text=True).stdout.splitlines():
        s, m, v = line.split()
        got[(s, m)] = int(v)
    for c, py in pairs.items():
        assert got[(c, "sizeof")] == ctypes.sizeof(py), c
        for f, _ in py._fields_:
            assert got[(c, f)] == getattr(py, f).offset, (c, f)


def test_step_rejects_bad_negative_regions(lib):
    # a negative flag other than 0 / 1
    a = _valid_args()
    arr = (gs.RegionDesc * 1)(gs.RegionDesc(0, 0, 2, 4, 1.0, 0, None, 0, 0x4000, 4, 0.0, 0.0, 2))
    a.n_regions = 1
    a.regions = ctypes.cast(arr, ctypes.POINTER(gs.RegionDesc))
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG
    # only negative regions and no full-frame cond: the positive branch is empty
    a = _valid_args()
    a.cond = 0
    arr = (gs.RegionDesc * 1)(gs.RegionDesc(0, 0, 2, 4, 1.0, 0, None, 0, 0x4000, 4, 0.0, 0.0, 1))
    a.n_regions = 1
    a.regions = ctypes.cast(arr, ctypes.POINTER(gs.RegionDesc))
    assert lib.gs_guided_step(ctypes.byref(a), None) == gs.GS_ERR_INVALID_ARG


def test_step_plan_checks_before_any_launch(lib):
    """gs_step_prepare answers like gs_guided_step's checks; gs_step_launch refuses an
    unprepared plan and a step index out of range before launching anything."""
    plan = gs.StepPlan()
    assert lib.gs_step_prepare(ctypes.byref(_valid_args()), None) == gs.GS_ERR_INVALID_ARG
    for field, value in (("B", 0), ("x", 0), ("n_sigmas", 1), ("n_regions", 17)):
        a = _valid_args()
        setattr(a, field, value)
        assert lib.gs_step_prepare(ctypes.byref(a), ctypes.byref(plan)) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_step_launch(ctypes.byref(gs.StepPlan()), 0, None) == gs.GS_ERR_INVALID_ARG
    assert lib.gs_step_launch(None, 0, None) == gs.GS_ERR_INVALID_ARG
    a = _valid_args()                                     # n_sigmas 5: steps 0 .. 3
    a.step = 99                                           # (ignored by the plan)
    assert lib.gs_step_prepare(ctypes.byref(a), ctypes.byref(plan)) == gs.GS_OK
    for step in (-1, 4, 1 << 30):
        assert lib.gs_step_launch(ctypes.byref(plan), step, None) == gs.GS_ERR_INVALID_ARG
