"""Host-only checks of the stream MHLA kernel's item order (no GPU).

``tests/sched_check.cpp`` includes the very header the kernel uses
(``csrc/stream_sched.h``) and, for each case, walks the whole item list:
every item once, every MIX item of a head after all of its SUM items, every
OUT item after all of its MIX items (the property that makes the kernel's
cross-CTA waits deadlock-free), and the gaps the host's lag choice reports.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "token_level_head_gb300", "csrc")

CASES = [  # heads, C, I, target gap (6 x 152 CTAs)
    (48, 32, 8, 912),     # the DiT-like workload: B8 x H6, N 4096, M 16
    (1, 1, 8, 912),
    (2, 8, 8, 912),
    (6, 32, 8, 912),
    (3, 5, 8, 912),
    (96, 48, 32, 912),
    (200, 32, 8, 912),
    (1, 64, 32, 912),
    (5000, 32, 8, 912),
]


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path_factory.mktemp("sched") / "sched_check")
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", CSRC, os.path.join(ROOT, "tests", "sched_check.cpp"), "-o", exe],
                   check=True)
    return exe


def run(exe, cases):
    args = [str(x) for c in cases for x in c]
    res = subprocess.run([exe, *args], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    return [tuple(map(int, line.split())) for line in res.stdout.split("\n") if line.strip()]


def test_every_item_once_and_dependencies_earlier(checker):
    out = run(checker, CASES)
    assert len(out) == len(CASES)
    for (heads, C, I, Dx, Do, E, worst), case in zip(out, CASES):
        assert (heads, C, I) == case[:3]
        assert E == heads * (2 * C + I)
        assert 0 <= Dx <= Do <= heads
        assert worst >= 1




def test_gap_targets(checker):
    out = {c[:3]: r for c, r in zip(CASES, run(checker, CASES))}
    # DiT-like: all SUM items before any OUT item (Do = heads) and the MIX
    # items half way, 769 positions (> 5 waves of 152 CTAs) on both sides
    heads, C, I, Dx, Do, E, worst = out[(48, 32, 8)]
    assert (Dx, Do, worst) == (24, 48, 769)
    # many heads: the target is reached with a bounded lag (L2 footprint)
    for key in ((200, 32, 8), (5000, 32, 8), (96, 48, 32)):
        heads, C, I, Dx, Do, E, worst = out[key]
        assert worst >= 912 and Do < 64
