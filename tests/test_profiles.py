"""The committed ncu summaries belong to the committed kernels: every entry of
profiles/traffic.json, and the source hash each summary under profiles/
states, equals bench.py's hash of that kernel's current sources.  A kernel
edit without a fresh capture fails here (bench.py then reports the traffic as
unknown rather than quoting stale counters)."""
import json
import os
import re

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")

# traffic.json key prefix / summary file prefix -> the sources bench.py hashes
SOURCES = {
    "split": bench.SPLIT_SOURCES,
    "toplp": bench.TOPLP_SOURCES,
    "gumbel": bench.GUMBEL_SOURCES,
    "penalty": bench.PENALTY_SOURCES,
    "spec_verify": bench.VERIFY_SOURCES,
    "smp": bench.KERNEL_SOURCES,
}


def sources_for_key(key):
    if ":" in key:
        return SOURCES[key.split(":")[0]]
    if key.startswith("verify"):
        return bench.VERIFY_SOURCES
    return bench.KERNEL_SOURCES


def traffic_entries():
    with open(os.path.join(PROFILES, "traffic.json")) as f:
        return sorted(json.load(f).items())


@pytest.mark.parametrize("key,entry", traffic_entries())
def test_traffic_entry_matches_current_sources(key, entry):
    assert entry["kernel_source_sha"] == bench.kernel_source_hash(sources_for_key(key)), key
    assert entry["dram_bytes_read_per_launch"] > 0
    assert "--clock-control none" in entry["command"]


def summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


@pytest.mark.parametrize("name", summaries())
def test_summary_states_the_current_source_hash(name):
    with open(os.path.join(PROFILES, name)) as f:
        text = f.read()
    shas = set(re.findall(r"sha `([0-9a-f]{16})`", text))
    assert len(shas) == 1, (name, shas)
    prefix = next(p for p in SOURCES if name.startswith(p + "_"))
    assert shas.pop() == bench.kernel_source_hash(SOURCES[prefix]), name
    # every ncu command quoted in a summary (indented code lines, joined over
    # their continuation backslashes) leaves the clocks alone
    joined = re.sub(r"\\\n\s*", " ", text)
    cmds = [l.strip() for l in joined.splitlines() if re.match(r"^ {4}ncu --", l)]
    assert cmds, name
    for cmd in cmds:
        assert "--clock-control none" in cmd, (name, cmd)
