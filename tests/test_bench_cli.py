"""bench.py's workload options and the seeded inputs they draw (CPU only)."""

import sys

import pytest
import torch

import bench
from bucketized_guidance_step_gb300.workloads import WORKLOADS, step_inputs


def _wl(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.workload_for(bench.parse_args())
    finally:
        sys.argv = old


def test_default_is_the_largest_workload():
    """The headline line times the throughput sweep (B=64, 16x128x128 bf16), the largest
    configuration that fits one GPU; the other target workloads follow in per_config."""
    wl = _wl()
    assert wl.name == "sweep_bf16_b64" and wl.sampler == "euler" and not wl.model_input
    assert wl.elements == max(w.elements for w in WORKLOADS)
    assert set(bench.TARGET_WORKLOADS) == {w.name for w in WORKLOADS[1:]}


def test_cpu_procs_default_to_host_cores():
    old = sys.argv
    sys.argv = ["bench.py"]
    try:
        args = bench.parse_args()
    finally:
        sys.argv = old
    assert args.cpu_procs == bench.host_cores() >= 1


def test_traffic_entries_split_read_and_write():
    for key, entry in bench.TRAFFIC.items():
        read, write, rev = entry
        assert read > 0 and write >= 0 and len(rev) == 16, key


def test_variant_names_and_fields():
    wl = _wl("--workload", "sweep_bf16_b64", "--sampler", "euler_ancestral", "--model-in",
             "--negative-regions", "1")
    assert wl.name == "sweep_bf16_b64@euler_ancestral@neg1@model_in"
    assert wl.sampler == "euler_ancestral" and wl.model_input and wl.negative_regions == 1
    wl = _wl("--workload", "bcg_bf16_b16", "--buckets", "4", "--batch", "8")
    assert wl.guidance.num_buckets == 4 and wl.B == 8 and wl.name == "bcg_bf16_b16@buckets4@B8"


@pytest.mark.parametrize("argv", [
    ("--workload", "bcg_bf16_b16", "--model-in"),                  # no inpaint
    ("--workload", "area_fp16_b8", "--buckets", "4"),              # scalar cfg
    ("--workload", "sweep_bf16_b64", "--negative-regions", "3"),   # no positive entry left
    ("--workload", "area_fp16_b8", "--negative-regions", "5"),     # more than its regions
])
def test_invalid_variants_exit(argv):
    with pytest.raises(SystemExit):
        _wl(*argv)


def test_algorithmic_bytes_of_the_variants():
    base = _wl("--workload", "sweep_bf16_b64")
    anc = _wl("--workload", "sweep_bf16_b64", "--sampler", "euler_ancestral", "--model-in")
    proto = step_inputs(base, 0, B=1).regions
    frame = 64 * 16 * 128 * 128 * 2
    assert bench.algorithmic_bytes(anc, proto) - bench.algorithmic_bytes(base, proto) == \
        frame + frame + 32 * 16 * 128 * 128 * 2        # noise, model input, fixed noise of 32


def test_sampler_inputs_are_seeded_and_distinct():
    import dataclasses
    wl = dataclasses.replace(WORKLOADS[3], sampler="euler_ancestral", model_input=True)
    a = step_inputs(wl, 2, B=2, C=2, H=8, W=8)
    b = step_inputs(wl, 2, B=2, C=2, H=8, W=8)
    assert torch.equal(a.fresh_noise, b.fresh_noise) and torch.equal(a.orig_noise, b.orig_noise)
    assert not torch.equal(a.fresh_noise, a.orig_noise)
    assert not torch.equal(a.fresh_noise, a.noise)
    plain = step_inputs(WORKLOADS[3], 2, B=2, C=2, H=8, W=8)
    assert plain.fresh_noise is None and plain.orig_noise is None
    assert torch.equal(plain.noise, a.noise)           # the other inputs do not move
    with pytest.raises(ValueError):
        step_inputs(dataclasses.replace(WORKLOADS[1], model_input=True), 0, B=1)


def test_binding_rejects_mismatched_sampler_tensors():
    """Shape checks of the Python binding run before any device pointer is taken."""
    from bucketized_guidance_step_gb300 import gs
    x = torch.zeros(2, 3, 4, 8)
    sig = torch.tensor([1.0, 0.0])
    with pytest.raises(ValueError, match="noise must have the shape"):
        gs.make_step_args(x, sigmas=sig, cond=x, noise=torch.zeros(2, 3, 4, 4),
                          sampler="euler_ancestral")
    with pytest.raises(ValueError, match="model_in_out must have the shape"):
        gs.make_step_args(x, sigmas=sig, cond=x, model_in_out=torch.zeros(1, 3, 4, 8))
    with pytest.raises(ValueError, match="orig_noise must have the shape"):
        gs.make_step_args(x, sigmas=sig, cond=x, orig_noise=torch.zeros(2, 3, 5, 8))


def test_kernel_hash_ignores_comments_only():
    """The traffic counters stay valid across comment edits, not across code edits."""
    a = bench._code_only('int f(int x) {  // doubles\n  /* the\n  value */ return 2 * x; }\n')
    b = bench._code_only('int f(int x) { return 2 * x; }  // twice x')
    c = bench._code_only('int f(int x) { return 3 * x; }')
    assert a == b != c
    assert bench._code_only('const char* s = "// kept"; // dropped') == 'const char* s = "// kept";'


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the oracle on host cores (no GPU) and prints one
    JSON line with the headline's metric and unit, marked as the reference, whose
    cpu_baseline and e2e carry the same value and no host-device bytes."""
    import json
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1", "--cpu-procs", "2"],
                         cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["B"] == 64 and d["config"]["workload"].startswith("sweep_bf16_b64")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
