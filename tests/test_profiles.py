"""The commands quoted in the profile summaries still run against this tree.

Every summary under profiles/ gives the ncu command that produced it. These
CPU checks keep those commands reproducible as the code moves: the bench
arguments parse with bench.py's own parser (and keep its warm-up rule), the
pytest selections name test files and functions that exist, each ncu command
leaves the clocks alone, and each kernel filter matches a kernel in csrc/.
"""
from __future__ import annotations

import glob
import os
import re
import shlex

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _commands(path):
    """The shell commands in the fenced blocks of one summary, continuations joined."""
    text = open(path).read()
    blocks = re.findall(r"^```[^\n]*\n(.*?)^```", text, flags=re.S | re.M)
    cmds = []
    for block in blocks:
        joined = re.sub(r"\\\n\s*", " ", block)
        cmds += [ln.strip() for ln in joined.splitlines() if ln.strip().startswith("ncu ")]
    return cmds


def _kernel_names():
    names = set()
    for src in glob.glob(os.path.join(ROOT, "w8a8_quantized_decode_gb300", "csrc", "*.cu*")):
        s = open(src).read()
        # __global__ void [__launch_bounds__(...)] name(
        names |= set(re.findall(
            r"__global__\s+void\s+(?:__launch_bounds__\((?:[^()]|\([^()]*\))*\)\s*)?(\w+)\s*\(",
            s))
    return names


def test_every_summary_quotes_a_command():
    assert PROFILES
    for p in PROFILES:
        assert _commands(p), f"{os.path.basename(p)} gives no ncu command"


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_profile_commands_are_current(path):
    import bench
    kernels = _kernel_names()
    assert kernels
    for cmd in _commands(path):
        argv = shlex.split(cmd)
        assert argv[0] == "ncu"
        i = argv.index("--clock-control")
        assert argv[i + 1] == "none", cmd
        # kernel filter: every alternative of the regex names a kernel of csrc/
        if "-k" in argv:
            pat = argv[argv.index("-k") + 1]
            assert pat.startswith("regex:"), cmd
            for alt in pat[len("regex:"):].split("|"):
                stem = re.match(r"[A-Za-z_][A-Za-z0-9_]*", alt).group(0)
                # a mangled name carries the identifier first, template args after
                stem = re.sub(r"I[LE].*$", "", stem)
                assert any(stem in k for k in kernels), f"{alt!r} matches no kernel"
        if "bench.py" in argv:
            args = bench.build_parser().parse_args(argv[argv.index("bench.py") + 1:])
            assert args.warmup >= 3, cmd
            assert args.impl == "ours", cmd
        elif "pytest" in argv:
            target = next(a for a in argv if a.startswith("tests/"))
            src = open(os.path.join(ROOT, target)).read()
            sel = argv[argv.index("-k") + 1]
            for word in re.findall(r"\btest_\w+", sel):
                assert f"def {word}(" in src, f"{word} not in {target}"
        else:
            raise AssertionError(f"unknown program in {cmd}")
