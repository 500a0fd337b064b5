"""A plain C client of libgs.so (CPU): the host entry points called from C through
include/gs.h alone, their results checked against the oracle.

This is how a non-Python user links the library; it checks that the header compiles
as C, that the exported symbols link, and that a C caller gets the same schedules,
bucket plans, latent slices and packings the oracle defines.
"""

import os
import shutil
import subprocess

import numpy as np
import pytest

from bucketized_guidance_step_gb300 import build, gs
from oracle import buckets as OB
from oracle import conds as OC
from oracle import schedules as OS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CLIENT = r"""
#include <stdio.h>
#include "gs.h"

int main(void) {
    printf("abi %d\n", (int)gs_abi_version());
    gs_schedule_desc d = {GS_SCHED_KARRAS, 10, 0.0292, 14.6146, 7.0, 1.0, -1, -1, 1, 1000,
                          0.00085, 0.012};
    float sig[16];
    int32_t n = 0, off = 0;
    if (gs_sigmas(&d, sig, 16, &n, &off) != GS_OK) return 1;
    printf("sigmas %d %d", (int)n, (int)off);
    for (int i = 0; i < n; ++i) printf(" %.9g", sig[i]);
    printf("\n");
    gs_curve_desc c = {0};
    c.kind = GS_CURVE_LINEAR; c.v0 = 2.0; c.v1 = 1.2;
    int32_t ids[50];
    float lut[50];
    if (gs_bucket_plan(50, 8, &c, NULL, ids, lut) != GS_OK) return 2;
    printf("plan");
    for (int i = 0; i < 50; ++i) printf(" %d:%.9g", (int)ids[i], lut[i]);
    printf("\n");
    gs_area a[2] = {{GS_AREA_PIXELS, 64, 128, 256, 512}, {GS_AREA_FRACTION, 0.25, 0.5, 0.5, 0.25}};
    gs_rect r[2];
    if (gs_areas_to_latent(a, 2, 128, 96, 8, r) != GS_OK) return 3;
    printf("areas %d %d %d %d %d %d %d %d\n", r[0].y0, r[0].x0, r[0].h, r[0].w, r[1].y0, r[1].x0,
           r[1].h, r[1].w);
    gs_cond_entry e[3] = {{32, 32, 3, 0}, {32, 32, 2, 0}, {64, 64, 1, 5}};
    gs_cond_chunk ch[8];
    int32_t nch = 0, ncall = 0;
    if (gs_pack_conds(e, 3, 4096, ch, 8, &nch, &ncall) != GS_OK) return 4;
    printf("pack %d", (int)ncall);
    for (int i = 0; i < nch; ++i) printf(" %d,%d,%d,%d", ch[i].call, ch[i].entry, ch[i].row0, ch[i].rows);
    printf("\n");
    printf("bad %d %s\n", (int)gs_bucket_plan(0, 8, &c, NULL, ids, lut),
           gs_status_string(GS_ERR_INVALID_ARG));
    return 0;
}
"""


def test_c_client_matches_oracle(repo_tmp):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    build.build()
    lib = gs.library_path()
    src = repo_tmp / "client.c"
    src.write_text(CLIENT)
    exe = repo_tmp / "client"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), lib,
                    "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    lines = {ln.split()[0]: ln.split()[1:] for ln in out.splitlines()}

    assert int(lines["abi"][0]) == gs.GS_ABI_VERSION
    n, off, *vals = lines["sigmas"]
    want, woff = OS.sigmas(OS.KARRAS, 10, sigma_min=0.0292, sigma_max=14.6146, rho=7.0,
                           force_full_denoise=True)
    assert int(n) == len(want) and int(off) == woff
    got = np.array([float(v) for v in vals], dtype=np.float32)
    wf = want.astype(np.float32)
    ulp = np.abs(got.view(np.int32).astype(np.int64) - wf.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1

    ids, lut = OB.plan(50, 8, OB.bucket_table(OB.linear_curve(2.0, 1.2), 8))
    pairs = [p.split(":") for p in lines["plan"]]
    assert [int(a) for a, _ in pairs] == ids.tolist()
    assert np.array_equal(np.array([float(b) for _, b in pairs], dtype=np.float32), lut)

    assert [int(v) for v in lines["areas"]] == \
        list(OC.area_to_latent(OC.PIXELS, 64, 128, 256, 512, 128, 96, 8)) + \
        list(OC.area_to_latent(OC.FRACTION, 0.25, 0.5, 0.5, 0.25, 128, 96))

    ncall, *chunks = lines["pack"]
    wn, wchunks = OC.pack_conds([(32, 32, 3, 0), (32, 32, 2, 0), (64, 64, 1, 5)], 4096)
    assert int(ncall) == wn
    assert [tuple(int(v) for v in c.split(",")) for c in chunks] == wchunks

    assert int(lines["bad"][0]) == gs.GS_ERR_INVALID_ARG
