"""Every ncu summary under profiles/ quotes the command that made it; those
commands must still run against the committed bench.py (its flags parse) and
name no file outside the repository (CPU)."""
from __future__ import annotations

import glob
import os
import re
import shlex

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _commands(path):
    """The shell commands inside the ``` blocks of a summary, with backslash
    continuations joined and trailing comments dropped."""
    text = open(path).read()
    cmds = []
    for block in re.findall(r"```\n(.*?)```", text, flags=re.S):
        joined = re.sub(r"\\\n\s*", " ", block)
        for line in joined.splitlines():
            line = line.split("#")[0].strip()
            if line:
                cmds.append(line)
    return cmds


def _bench_args(cmd):
    """The arguments of each `python bench.py ...` inside a command (plain, or
    wrapped by ncu)."""
    words = shlex.split(cmd)
    out = []
    for i, w in enumerate(words):
        if w == "bench.py" and i > 0 and words[i - 1].startswith("python"):
            out.append(words[i + 1:])
    return out


def test_every_summary_quotes_its_command():
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))
    assert paths
    for p in paths:
        assert _commands(p), f"{os.path.basename(p)} quotes no command"


def test_quoted_bench_commands_parse_with_the_committed_flags():
    parser = bench.build_parser()
    seen = 0
    for p in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for cmd in _commands(p):
            for args in _bench_args(cmd):
                parser.parse_args(args)  # exits (SystemExit) on an unknown flag
                seen += 1
    assert seen > 0


def test_quoted_commands_read_no_path_outside_the_repository():
    for p in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for cmd in _commands(p):
            for w in shlex.split(cmd):
                assert not w.startswith("/"), f"{os.path.basename(p)}: absolute path {w}"
