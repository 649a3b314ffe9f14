"""The committed ncu summaries under profiles/ each give the full command
that made them, with the clocks left alone, and that command runs committed
files only: bench.py with options it accepts."""
import glob
import os
import re
import shlex
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _commands(text):
    """The indented command block of a summary, continuation lines joined."""
    block, cmds = [], []
    for line in text.splitlines():
        if line.startswith("    ") and line.strip():
            block.append(line.strip())
        elif block:
            cmds.append(" ".join(block).replace("\\ ", " "))
            block = []
    if block:
        cmds.append(" ".join(block).replace("\\ ", " "))
    return [c for c in cmds if c.startswith("ncu ")]


def _bench_options():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True,
                       text=True, cwd=ROOT, timeout=120)
    assert r.returncode == 0, r.stderr
    return set(re.findall(r"(--[a-z0-9-]+)", r.stdout))


def test_every_summary_names_its_command():
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert files
    opts = _bench_options()
    for f in files:
        cmds = _commands(open(f).read())
        assert cmds, f"{f}: no ncu command"
        for c in cmds:
            words = shlex.split(c)
            assert "--clock-control" in words and words[words.index("--clock-control") + 1] == "none", f
            i = words.index("python")
            assert words[i + 1] == "bench.py" and os.path.exists(os.path.join(ROOT, words[i + 1])), f
            for w in words[i + 2:]:
                if w.startswith("--"):
                    assert w in opts, f"{f}: bench.py has no option {w}"
