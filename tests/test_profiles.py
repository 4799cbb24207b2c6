"""The committed profile summaries stay runnable and consistent (CPU only).

Every command quoted under profiles/ runs committed files: bench.py with one
of its named profile cases and its other flags, with --clock-control none on
every ncu command.  Every DRAM-byte record in profiles/traffic.json names an
existing source file that defines the kernel it names, and its command."""
import glob
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _bench_cases():
    text = open(os.path.join(ROOT, "bench.py")).read()
    m = re.search(r"PROFILE_CASES\s*=\s*\(([^)]*)\)", text)
    assert m, "bench.py defines PROFILE_CASES"
    return set(re.findall(r'"([a-z0-9_]+)"', m.group(1)))


def _texts():
    """Each summary and each recorded command as one line (wrapped lines and
    continuation backslashes joined)."""
    out = []
    for path in sorted(glob.glob(os.path.join(PROFILES, "*.md"))):
        text = open(path).read().replace("\\\n", " ").replace("\n", " ")
        out.append((os.path.basename(path), re.sub(r"\s+", " ", text)))
    rec = json.load(open(os.path.join(PROFILES, "traffic.json")))
    for k, cmd in rec["commands"].items():
        out.append(("traffic.json:" + k, cmd))
    return out


def test_profile_commands_run_committed_files():
    cases = _bench_cases()
    texts = _texts()
    n_ncu = 0
    for where, text in texts:
        for case in re.findall(r"--profile-case ([a-z0-9_]+)", text):
            assert case in cases, (where, case)
        for script in re.findall(r"python ([\w./-]+\.py)", text):
            assert os.path.exists(os.path.join(ROOT, script)), (where, script)
        # every ncu run (ncu, then options each with at most one value, then
        # the profiled program) leaves the clocks alone; ncu -i only reads a
        # report; "ncu" in prose is not followed by that shape
        for opts in _ncu_commands(text):
            if opts[:1] == ["-i"]:
                continue
            n_ncu += 1
            assert "--clock-control" in opts and opts[opts.index("--clock-control") + 1] == "none", \
                (where, " ".join(opts)[:120])
    assert n_ncu >= 5


def _ncu_commands(text):
    """The option lists of the ncu commands in text."""
    toks = text.replace("`", " ").split()
    for i, t in enumerate(toks):
        if t != "ncu":
            continue
        j, opts = i + 1, []
        while j < len(toks) and toks[j].startswith("-"):
            opts.append(toks[j])
            j += 1
            if j < len(toks) and not toks[j].startswith("-") and toks[j] != "python":
                opts.append(toks[j])
                j += 1
        if opts and j < len(toks) and toks[j] == "python":
            yield opts


@pytest.mark.parametrize("kind", ["index_score", "select_topk", "sparse_attn", "sparse_attn_fp8",
                                  "append_token", "hot_plan", "sparse_attn_planned"])
def test_traffic_records_name_real_kernels(kind):
    rec = json.load(open(os.path.join(PROFILES, "traffic.json")))
    r = rec["kernels"][kind]
    src = os.path.join(ROOT, r["source"])
    assert os.path.exists(src), r["source"]
    assert re.search(r"\b%s\s*\(" % re.escape(r["kernel"]), open(src).read()), (kind, r["kernel"])
    assert r["dram_read_bytes"] >= 0 and r["dram_write_bytes"] >= 0
    assert len(r["sha256"]) == 64
