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
