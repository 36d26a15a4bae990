"""The profile summaries under profiles/ quote the commands that produced
their figures.  Every `python bench.py ...` in them must still parse with the
bench's own argument parser (no GPU, nothing is run)."""

import glob
import os
import re
import shlex
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench_commands():
    cmds = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read().replace("\\\n", " ")
        for m in re.finditer(r"python bench\.py([^`\n>&|]*)", text):
            cmds.append((os.path.basename(path), shlex.split(m.group(1))))
    return cmds


def test_profile_commands_parse_with_the_bench():
    sys.path.insert(0, ROOT)
    import bench
    cmds = _bench_commands()
    assert cmds, "no bench command quoted under profiles/"
    for name, argv in cmds:
        args = bench.parse(argv)
        assert args.impl == "gb300", name
        assert args.steps >= 1 and args.warmup >= 1, name
