"""The ncu summaries under profiles/: each names the command that made it, and
that command runs only files of this repository (no scratch scripts)."""

import os
import re
import subprocess

from tests.conftest import ROOT

PROFILES = os.path.join(ROOT, "profiles")


def tracked_files():
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    if out.returncode != 0:
        return None
    return set(out.stdout.split())


def test_every_profile_gives_commands_that_run_committed_files():
    tracked = tracked_files()
    names = sorted(f for f in os.listdir(PROFILES) if f.endswith((".md", ".txt")))
    assert names, "no profile summaries"
    for name in names:
        text = open(os.path.join(PROFILES, name)).read()
        assert "_work/" not in text, f"{name} refers to a scratch file"
        scripts = re.findall(r"\bpython3?\s+(?:-m\s+\S+\s+)?([\w./-]+\.py)\b", text)
        assert scripts, f"{name} gives no python command"
        for s in scripts:
            assert os.path.exists(os.path.join(ROOT, s)), f"{name}: {s} does not exist"
            if tracked is not None:
                assert s in tracked, f"{name}: {s} is not committed"
        # the profiler's clocks are left alone on every ncu command
        for line in text.splitlines():
            if line.strip().startswith("ncu "):
                block = text[text.index(line):text.index(line) + 400]
                assert "--clock-control none" in block, f"{name}: ncu without --clock-control none"
