"""The bench commands quoted in the ncu summaries under profiles/ parse with
today's bench.py (CPU).

Each summary gives the command that produced its figures; a renamed or
removed bench option would leave a command nobody can rerun.  The
commands are joined across backslash line continuations, and every
`python bench.py ...` in them is parsed by bench.py's own argument parser."""
import glob
import os
import re
import shlex
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_commands():
    cmds = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read().replace("\\\n", " ")
        for line in text.splitlines():
            for m in re.finditer(r"python bench\.py([^\"`\n]*)", line):
                cmds.append((os.path.basename(path), m.group(1).strip()))
    return cmds


def test_profiles_quote_bench_commands():
    assert len(bench_commands()) >= 5


@pytest.mark.parametrize("name,args", bench_commands())
def test_quoted_bench_command_parses(name, args):
    saved = sys.argv
    try:
        sys.argv = ["bench.py"] + shlex.split(args)
        import bench
        bench.parse()  # argparse exits on an unknown option or a bad value
    except SystemExit as ex:
        pytest.fail(f"{name}: 'python bench.py {args}' does not parse ({ex})")
    finally:
        sys.argv = saved
