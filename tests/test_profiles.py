"""The ncu summaries under profiles/ stay reproducible with the committed files
(CPU): every command names a workload bench.py still knows, every ncu command
leaves the GPU's clocks alone (--clock-control none) and captures one kernel
a few launches at a time (or is the one-pass launch list), and the DRAM traffic
table the bench reads names workloads that exist."""
import json
import os
import re

import pytest

from sliding_window_sink_bias_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
SUMMARIES = sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def _commands(text):
    """The fenced command blocks of a summary, continuation lines joined."""
    blocks = re.findall(r"```\n(.*?)```", text, flags=re.S)
    return [b.replace("\\\n", " ") for b in blocks]


@pytest.mark.parametrize("name", SUMMARIES)
def test_summary_command_is_reproducible(name):
    with open(os.path.join(PROFILES, name)) as f:
        text = f.read()
    cmds = _commands(text)
    assert cmds, f"{name}: no command block"
    for block in cmds:
        for wl in re.findall(r"--workload ([a-z0-9_]+)", block):
            assert wl in synth.WORKLOADS, f"{name}: unknown workload {wl}"
        for line in block.splitlines():
            if not re.search(r"(^|\s)ncu\s", line) or " -i " in line:
                continue  # not a capture (or the export of a saved report)
            assert "--clock-control none" in line, f"{name}: {line.strip()}"
            if "--set full" in line or "--section" in line:
                # a full capture: one kernel, a few launches
                assert re.search(r"\s-k\s+\S+", line), f"{name}: no -k in {line.strip()}"
                m = re.search(r"\s-c\s+(\d+)", line)
                assert m and int(m.group(1)) <= 3, f"{name}: -c in {line.strip()}"
            else:
                # the launch list: one metric, one pass per launch
                assert "--metrics gpu__time_duration.sum" in line, f"{name}: {line.strip()}"


def test_traffic_table_names_known_workloads():
    with open(os.path.join(PROFILES, "dram_traffic.json")) as f:
        tab = json.load(f)
    for key, e in tab.items():
        assert e["workload"] in synth.WORKLOADS, key
        assert e["kernel"] in ("band", "causal", "decode"), key
        assert e["dram_bytes_per_launch"] > 0 and len(e["sha256"]) == 64, key
