"""The bench commands that the ncu summaries under profiles/ give as their
source still parse with bench.py's own options and name existing workloads, so
every summary can be reproduced from committed files."""

import pathlib
import re
import shlex

import bench
import synthetic

PROFILES = pathlib.Path(__file__).resolve().parent.parent / "profiles"


def _bench_commands():
    for path in sorted(PROFILES.glob("*.md")):
        text = re.sub(r"\\\n\s*", " ", path.read_text())   # shell line continuations
        for m in re.finditer(r"python bench\.py([^\n`]*)", text):
            yield path.name, m.group(1)


def test_every_profile_names_its_command():
    for path in sorted(PROFILES.glob("*.md")):
        text = path.read_text()
        assert "ncu " in text or "python bench.py" in text, path.name


def test_profile_bench_commands_parse():
    parser = bench.make_parser()
    n = 0
    for name, argstr in _bench_commands():
        args = parser.parse_args(shlex.split(argstr))
        assert args.workload in synthetic.CONFIGS, (name, args.workload)
        for w in filter(None, args.also.split(",")):
            assert w in synthetic.CONFIGS, (name, w)
        n += 1
    assert n >= 6


def test_profile_ncu_commands_leave_the_clocks_alone():
    n = 0
    for path in sorted(PROFILES.glob("*.md")):
        text = re.sub(r"\\\n\s*", " ", path.read_text())
        for line in text.splitlines():
            if re.match(r"\s*ncu\s+-", line):
                assert "--clock-control none" in line, (path.name, line.strip()[:80])
                n += 1
    assert n >= 6
