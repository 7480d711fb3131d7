"""Consistency of the committed ncu summaries (CPU only).

- Every ncu command in profiles/ leaves the GPU clocks alone
  (`--clock-control none`).
- profiles/ holds text summaries and traffic.json, nothing that runs.
- Each traffic.json entry names an existing summary and kernel source, with
  positive byte counts; the bench reports an entry only while its source hash
  matches, and reports nothing for a stale hash.
"""
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def _ncu_commands(text):
    """The ncu invocations in a summary's code blocks (continuation lines
    joined); reading a saved report (`ncu -i`) is not a capture."""
    blocks = re.findall(r"```[^\n]*\n(.*?)```", text, flags=re.S)
    cmds = []
    for b in blocks:
        joined = re.sub(r"\\\n\s*", " ", b)
        for ln in joined.splitlines():
            for part in re.split(r"&&|;", ln):
                part = part.strip()
                if re.match(r"ncu\s", part) and not re.match(r"ncu\s+-i\s", part):
                    cmds.append(part)
    return cmds


def test_profiles_hold_text_only():
    for f in os.listdir(PROFILES):
        assert f.endswith(".md") or f == "traffic.json", f"unexpected file in profiles/: {f}"


@pytest.mark.parametrize("name", _summaries())
def test_ncu_commands_leave_clocks_alone(name):
    text = open(os.path.join(PROFILES, name)).read()
    cmds = _ncu_commands(text)
    assert cmds, f"{name}: no ncu command recorded"
    for c in cmds:
        assert "--clock-control none" in c, f"{name}: ncu command without --clock-control none: {c}"


def test_traffic_entries_are_well_formed():
    d = json.load(open(os.path.join(PROFILES, "traffic.json")))
    entries = {k: v for k, v in d.items() if not k.startswith("_")}
    assert entries
    for k, v in entries.items():
        assert os.path.exists(os.path.join(PROFILES, v["summary"])), k
        assert os.path.exists(os.path.join(ROOT, "mxfp8_block_scaled_gb300", "csrc", v["source"])), k
        assert re.fullmatch(r"[0-9a-f]{16}", v["source_sha256_16"]), k
        counts = [v[f] for f in ("bytes_per_step", "bytes_per_launch") if f in v]
        assert counts and all(isinstance(c, int) and c > 0 for c in counts), k


def test_stale_traffic_is_not_reported(tmp_path, monkeypatch):
    import bench
    src_dir = tmp_path / "mxfp8_block_scaled_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (src_dir / "k.cu").write_text("kernel v2\n")
    (tmp_path / "profiles").mkdir()
    import hashlib
    h_old = hashlib.sha256(b"kernel v1\n").hexdigest()[:16]
    h_new = hashlib.sha256(b"kernel v2\n").hexdigest()[:16]
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "stale": {"bytes_per_step": 123, "source": "k.cu", "source_sha256_16": h_old, "summary": "x.md"},
        "fresh": {"bytes_per_step": 456, "source": "k.cu", "source_sha256_16": h_new, "summary": "x.md"}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("stale") is None
    assert bench.profile_traffic("fresh") == 456
    assert bench.profile_traffic("absent") is None
