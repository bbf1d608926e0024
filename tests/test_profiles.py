"""The profile summaries under profiles/ (CPU): every command they record runs a
committed script with arguments that script accepts, every ncu command leaves
the clocks alone (--clock-control none), and the traffic record matches the
scorer source it was captured from, or bench.py reports no traffic."""
import glob
import json
import os
import re
import shlex
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _commands():
    out = []
    for path in glob.glob(os.path.join(ROOT, "profiles", "*")):
        text = open(path).read()
        if path.endswith(".json"):
            text = json.loads(text).get("source", "")
        text = text.replace("\\\n", " ")
        out += [(path, l.strip()) for l in text.splitlines() if "python " in l or "ncu " in l]
    return out


def test_profile_commands_run_committed_scripts_with_known_flags(monkeypatch):
    import bench
    cmds = _commands()
    assert cmds
    for path, line in cmds:
        if "ncu " in line and "-i " not in line:
            assert "--clock-control none" in line, (path, line)
        m = re.search(r"python (\S+\.py)([^()]*)", line)
        if not m:
            continue
        script, args = m.group(1), shlex.split(m.group(2))
        assert os.path.exists(os.path.join(ROOT, script)), (path, script)
        if script == "bench.py":
            monkeypatch.setattr(sys, "argv", ["bench.py"] + args)
            bench.parse_args()        # exits on an unknown flag


def test_traffic_record_matches_the_scorer_source():
    import bench
    d = json.load(open(os.path.join(ROOT, "profiles", "score_kernel_traffic.json")))
    assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"]
    if d["kernel_sha"] == bench.score_kernel_sha():
        assert bench.ncu_traffic(d["workload"]) == d["dram_bytes_per_launch"]
    else:
        assert bench.ncu_traffic(d["workload"]) is None
