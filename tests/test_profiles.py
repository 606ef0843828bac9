"""The ncu summaries under profiles/: every recorded ncu command leaves the
GPU clocks alone (--clock-control none) and captures a bounded number of
launches; every summary that feeds bench.py's roofline traffic names the
kernel sources its hash covers and a positive byte count."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _ncu_commands(text):
    """The ncu command lines of a summary, continuation lines joined."""
    joined = re.sub(r"\\\n\s*", " ", text)
    return [ln.strip() for ln in joined.splitlines() if re.match(r"^\s*ncu\s", ln)]


def test_every_ncu_command_keeps_the_clocks_and_bounds_its_launches():
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert paths
    seen = 0
    for p in paths:
        for cmd in _ncu_commands(open(p, encoding="utf-8").read()):
            seen += 1
            assert "--clock-control none" in cmd, (os.path.basename(p), cmd)
            assert re.search(r"\s-c\s+\d+", cmd), (os.path.basename(p), cmd)
            if "--set full" in cmd:
                # full captures: one kernel, at most three launches
                assert re.search(r"\s-k\s+\S+", cmd), (os.path.basename(p), cmd)
                assert int(re.search(r"\s-c\s+(\d+)", cmd).group(1)) <= 3, cmd
    assert seen >= len(paths)


def test_traffic_summaries_are_complete():
    import bench
    for config, (name, sources) in bench.TRAFFIC_SUMMARIES.items():
        text = open(os.path.join(ROOT, "profiles", name), encoding="utf-8").read()
        assert re.search(r"kernel_sources_sha256:\s*[0-9a-f]{64}", text), name
        m = re.search(r"dram_bytes_per_launch_full_workload:\s*(\d+)", text)
        assert m and int(m.group(1)) > 0, name
        for src in sources:
            assert f"`{src}`" in text, (name, src)
