"""The ncu summaries under profiles/: each names the command that made it, that
command runs files of this repository with arguments they accept, every capture
sets --clock-control none, and the traffic table bench.py reads points at them."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
SUMMARIES = sorted(f for f in os.listdir(PROFILES) if f.endswith(".md") and f != "dram_traffic.md")


def _command(text):
    """The indented command block under the 'Command' line, joined over its continuations."""
    lines = text.splitlines()
    start = next(i for i, line in enumerate(lines) if line.startswith("Command"))
    block = []
    for line in lines[start + 1:]:
        if line.startswith("    "):
            block.append(line.strip().rstrip("\\").strip())
        elif block:
            break
    return " ".join(block)


@pytest.mark.parametrize("name", SUMMARIES)
def test_summary_names_a_runnable_command(name):
    text = open(os.path.join(PROFILES, name)).read()
    cmd = _command(text)
    assert cmd.startswith("ncu "), cmd
    assert "--clock-control none" in cmd
    py = cmd[cmd.index(" python ") + len(" python "):].split()
    if py[0] == "-m":
        module = py[1]
        path = os.path.join(ROOT, *module.split(".")) + ".py"
        assert os.path.exists(path), module
        args = py[2:]
        target = ["-m", module]
    else:
        assert os.path.exists(os.path.join(ROOT, py[0])), py[0]
        args = py[1:]
        target = [py[0]]
    # the script accepts these arguments (argument parsing only: --help after them exits before any work)
    r = subprocess.run([sys.executable] + target + args + ["--help"], cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, r.stderr[-500:]


def test_traffic_table_rows_point_at_summaries():
    rows = [line for line in open(os.path.join(PROFILES, "dram_traffic.md")) if line.startswith("| traffic:")]
    assert rows
    for line in rows:
        parts = [p.strip() for p in line.strip().strip("|").split("|")]
        assert int(parts[3]) > 0, line
        ref = re.match(r"([\w.]+\.md)", parts[4]).group(1)
        assert ref in SUMMARIES, ref
