"""Host-side bookkeeping of bench.py that needs no GPU: which committed ncu
counters the bench line may quote, and how it reads them."""
import os
import shutil

import bench


def test_fused_kernel_sources_exist():
    for rel in bench.FUSED_DECODE_SOURCES:
        assert os.path.isfile(os.path.join(bench.ROOT, rel)), rel


def test_fused_kernel_sources_cover_its_includes():
    # every project header the fused kernel's translation unit pulls in, and
    # every header of the host file that launches it, is part of the digest
    import re
    csrc = os.path.join(bench.ROOT, "quantized_routed_expert_gb300", "csrc")
    listed = {os.path.basename(p) for p in bench.FUSED_DECODE_SOURCES}
    todo, seen = ["decode_fused.cu", "decode.cu", "moe_api.cu"], set()
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.add(f)
        path = os.path.join(csrc, f)
        if not os.path.isfile(path):
            path = os.path.join(bench.ROOT, "include", f)
        with open(path) as fh:
            for inc in re.findall(r'^#include "([^"]+)"', fh.read(), re.M):
                todo.append(inc)
    assert seen <= listed, seen - listed


def test_traffic_is_quoted_only_for_the_profiled_sources(tmp_path, monkeypatch):
    prof = os.path.join(bench.ROOT, "profiles", bench.PROFILE_DECODE_FUSED)
    got = bench.profiled_traffic(bench.PROFILE_DECODE_FUSED, 1)
    with open(prof) as f:
        head = dict(ln.split(": ", 1) for ln in f.read().splitlines()[:4] if ": " in ln)
    if head.get("sources_digest") == bench.sources_digest():
        assert got is not None and got["dram_bytes_per_launch"] == float(head["dram_bytes_per_launch"])
    else:
        assert got is None
    # another token count, or sources edited since the capture: no figure
    assert bench.profiled_traffic(bench.PROFILE_DECODE_FUSED, 2) is None
    root = tmp_path / "repo"
    for rel in bench.FUSED_DECODE_SOURCES + ("profiles/" + bench.PROFILE_DECODE_FUSED,):
        dst = root / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.sources_digest() == head.get("sources_digest") or got is None
    with open(root / bench.FUSED_DECODE_SOURCES[0], "a") as f:
        f.write("\n// edited\n")
    assert bench.profiled_traffic(bench.PROFILE_DECODE_FUSED, 1) is None
