"""Source hygiene (CPU only): the committed code, comments and docstrings
stand on their own.  They cite the page by its title and sections, never
this build's own working files, paths or tooling, and nothing committed
reads the uncommitted working folder."""
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# names a committed source file must not contain (case-insensitive); the
# .md documents are exempt (they are where such files are named)
FORBIDDEN = [r"paper\.md", r"north_star", r"baseline\.json", r"/root/", r"gpurun", r"_work/",
             r"survey\.md", r"verdict\.md", r"advice\.md", r"design\.md", r"\bround \d+\b"]


def _sources():
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    if out.returncode != 0:  # not a checkout: walk the tree instead
        files = []
        for d, _, fs in os.walk(ROOT):
            if "/." in d or "_build" in d or "/_work" in d:
                continue
            files += [os.path.relpath(os.path.join(d, f), ROOT) for f in fs]
    else:
        files = out.stdout.split()
    exts = (".py", ".cu", ".cuh", ".h", ".c", ".ini", ".sh")
    return [f for f in files if f.endswith(exts) and os.path.exists(os.path.join(ROOT, f))]


def test_sources_name_no_working_files_or_tooling():
    pat = re.compile("|".join(FORBIDDEN), re.IGNORECASE)
    bad = []
    for f in _sources():
        if f == os.path.join("tests", "test_hygiene.py"):
            continue
        for n, line in enumerate(open(os.path.join(ROOT, f), errors="replace"), 1):
            if pat.search(line):
                bad.append(f"{f}:{n}: {line.strip()[:100]}")
    assert not bad, "\n".join(bad)

