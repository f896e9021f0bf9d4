"""The ncu summaries under profiles/ (CPU only): text files, each giving the
command that produced it. Every ncu command leaves the GPU clocks alone
(--clock-control none) and profiles the committed bench.py, nothing else."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*")))


def test_profiles_are_text_summaries():
    assert PROFILES
    for p in PROFILES:
        assert os.path.splitext(p)[1] in (".md", ".txt"), p
        assert os.path.getsize(p) < 64 * 1024, p


def test_every_summary_gives_its_ncu_command():
    for p in PROFILES:
        text = open(p).read()
        blocks = re.findall(r"```\n(.*?)```", text, flags=re.S)
        cmds = [b for b in blocks if "ncu " in b]
        assert cmds, f"{os.path.basename(p)}: no ncu command"
        for c in cmds:
            joined = c.replace("\\\n", " ")
            for line in joined.splitlines():
                if "ncu " in line:
                    assert "--clock-control none" in line, f"{os.path.basename(p)}: {line}"
                    assert "python bench.py" in line, f"{os.path.basename(p)}: {line}"
            assert "_work" not in c and "gpurun " not in c, os.path.basename(p)


def _ncu_lines(text):
    for b in re.findall(r"```\n(.*?)```", text, flags=re.S):
        for line in b.replace("\\\n", " ").splitlines():
            if "ncu " in line and " -i " not in line:
                yield line[line.index("ncu "):]


def test_captures_beyond_the_launch_list_stay_small():
    """A capture that collects more than gpu__time_duration.sum (more metrics,
    sections or sets) takes one kernel by its exact name, at most three
    launches, on a reduced case (a token and expert count given to bench.py);
    only the one-pass launch list may run on the full-size workload."""
    for p in PROFILES:
        for line in _ncu_lines(open(p).read()):
            m = re.search(r"--metrics\s+(\S+)", line)
            time_only = (m is not None and m.group(1) == "gpu__time_duration.sum"
                         and "--set" not in line and "--section" not in line)
            if time_only:
                continue
            name = os.path.basename(p)
            k = re.search(r"\s-k\s+(\S+)", line)
            assert k and not k.group(1).startswith("regex:"), f"{name}: one kernel by its exact name: {line}"
            c = re.search(r"\s-c\s+(\d+)", line)
            assert c and int(c.group(1)) <= 3, f"{name}: at most three launches: {line}"
            assert "--tokens" in line and "--experts" in line, f"{name}: a reduced case: {line}"
