"""The oracle's pins catch planted mistakes (CPU).

Each case copies oracle/ and the pin tests (tests/test_oracle_*.py, which import only
oracle/) into a scratch folder, plants one plausible mistake in the copy -- a swapped
operand, a dropped term, an off-by-one edge, a wrong branch -- and runs the pins of the
mutated module there in a separate process, which must fail (a pin run that does not
finish within 30 seconds, e.g. a packing loop that no longer advances, counts as failing).
The unmodified copy must pass.
"""

import glob
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (file, original text, planted text)
MUTATIONS = [
    ("step.py", "u + s * (pos - u)", "pos + s * (u - pos)"),
    ("step.py", "(h - rows) / F", "(h - rows - 1) / F"),
    ("step.py", "if x0 + w < W:", "if x0 + w <= W:"),
    ("step.py", "    return x + (sigma_next - sigma) * d", "    return x + (sigma - sigma_next) * d"),
    ("step.py", "m * pred + (1.0 - m) * np.asarray(orig", "(1.0 - m) * pred + m * np.asarray(orig"),
    ("step.py", "        wsum += 1.0", "        wsum += 0.0"),
    ("step.py", "np.where(on, wgt * out, 0.0)", "np.where(on, wgt * out * wgt, 0.0)"),
    ("step.py", "return r.t_start <= p < r.t_end", "return r.t_start < p < r.t_end"),
    ("step.py", "sigma ** 2 - sigma_next ** 2)", "sigma_next ** 2 - sigma ** 2)"),
    ("step.py", "np.sqrt(np.maximum(sigma_next ** 2 - up ** 2, 0.0))",
     "np.sqrt(np.maximum(sigma_next ** 2 + up ** 2, 0.0))"),
    ("step.py", "(down.reshape(B, 1, 1, 1) - sigma) * d", "(down.reshape(B, 1, 1, 1) + sigma) * d"),
    ("step.py", "up.reshape(B, 1, 1, 1) * \\\n", "down.reshape(B, 1, 1, 1) * \\\n"),
    ("step.py", "out = m * x_next + (1.0 - m) * noised", "out = m * x_next + m * noised"),
    ("step.py", "+ sn * np.asarray(orig_noise", "+ np.asarray(orig_noise"),
    ("step.py", "ok &= sigma_next >= 0.0", "ok &= sigma_next > 0.0"),
    ("step.py", "if not r.negative]", "]"),
    ("step.py", "unc = positive_branch(B, C, H, W, cond=uncond,", "unc = positive_branch(B, C, H, W, cond=None,"),
    ("schedules.py", "(a + t * (b - a)) ** rho", "(a + t * (b - a)) ** (1.0 / rho)"),
    ("schedules.py", "offset = total - steps", "offset = total - steps - 1"),
    ("schedules.py", "w = t - lo", "w = hi - t"),
    ("buckets.py", "(b + 0.5) / num_buckets", "b / num_buckets"),
    ("buckets.py", "min(b, num_buckets - 1)", "min(b, num_buckets)"),
    ("buckets.py", "((1.0 - p) / (1.0 - apex))", "(p / (1.0 - apex))"),
    ("buckets.py", "f = p * num_buckets - b", "f = p * num_buckets - b - 0.5"),
    ("mask.py", "(j + 0.5) * scale - 0.5", "j * scale"),
    ("mask.py", "(np.uint32(nz[-1] + 1) << np.uint32(16))", "(np.uint32(nz[-1]) << np.uint32(16))"),
    ("mask.py", "np.uint32(nz[0]) | ", "np.uint32(nz[0] + 1) | "),
    ("conds.py", "top = max(math.floor(ly0), 0)", "top = max(math.ceil(ly0), 0)"),
    ("conds.py", "bottom = min(math.ceil(ly0 + lh), H)", "bottom = min(math.floor(ly0 + lh), H)"),
    ("conds.py", "lx0, lw = vals[1] * float(W), vals[3] * float(W)",
     "lx0, lw = vals[1] * float(H), vals[3] * float(W)"),
    ("conds.py", "cap = max(1, budget // (h * w))", "cap = max(1, budget // h)"),
    ("conds.py", "if cur is None or cur[1] >= cap:", "if cur is None or cur[1] > cap:"),
    ("conds.py", "key = (h, w, options)", "key = (h, w)"),
]


# the pin file of each oracle module
PINS = {"step.py": "test_oracle_step.py", "schedules.py": "test_oracle_schedules.py",
        "buckets.py": "test_oracle_buckets.py", "mask.py": "test_oracle_mask.py",
        "conds.py": "test_oracle_conds.py"}


def _copy(dst):
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    open(os.path.join(dst, "tests", "__init__.py"), "w").close()
    for p in glob.glob(os.path.join(ROOT, "tests", "test_oracle_*.py")):
        if not p.endswith("test_oracle_mutations.py"):
            shutil.copy(p, os.path.join(dst, "tests", os.path.basename(p)))


def _pins_pass(dst, pin_file) -> bool:
    try:
        r = subprocess.run([sys.executable, "-m", "pytest", os.path.join("tests", pin_file),
                            "-x", "-q", "-p", "no:cacheprovider", "--rootdir", dst],
                           cwd=dst, capture_output=True, text=True, timeout=30)
    except subprocess.TimeoutExpired:
        return False
    return r.returncode == 0


@pytest.mark.parametrize("pin_file", sorted(set(PINS.values())))
def test_unmodified_copy_passes(repo_tmp, pin_file):
    _copy(str(repo_tmp))
    assert _pins_pass(str(repo_tmp), pin_file)


@pytest.mark.parametrize("f,old,new", MUTATIONS, ids=[f"{m[0]}:{i}" for i, m in
                                                     enumerate(MUTATIONS)])
def test_planted_mistake_is_caught(repo_tmp, f, old, new):
    _copy(str(repo_tmp))
    path = os.path.join(str(repo_tmp), "oracle", f)
    src = open(path).read()
    assert src.count(old) == 1, f"mutation anchor not found once in {f}: {old!r}"
    open(path, "w").write(src.replace(old, new))
    assert not _pins_pass(str(repo_tmp), PINS[f]), \
        f"planted mistake survived: {f}: {old!r} -> {new!r}"
