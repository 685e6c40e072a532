"""Host-side bookkeeping of bench.py that needs no GPU: which committed ncu
counters the bench line may quote, and how it reads them."""
import json
import os
import re
import shutil

import pytest

import bench

KERNELS = [(bench.FUSED_DECODE_SOURCES, ["decode_fused.cu", "decode.cu", "moe_api.cu"]),
           (bench.LAYERS_DECODE_SOURCES, ["decode_layers.cu", "decode.cu", "moe_api.cu"])]


@pytest.mark.parametrize("files,roots", KERNELS)
def test_kernel_sources_exist_and_cover_their_includes(files, roots):
    # every project header the kernel's translation unit pulls in, and every
    # header of the host files that launch it, is part of the digest
    for rel in files:
        assert os.path.isfile(os.path.join(bench.ROOT, rel)), rel
    csrc = os.path.join(bench.ROOT, "quantized_routed_expert_gb300", "csrc")
    listed = {os.path.basename(p) for p in files}
    todo, seen = list(roots), set()
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


def test_committed_profiles_are_machine_readable():
    for name in (bench.PROFILE_DECODE_FUSED, bench.PROFILE_DECODE_LAYERS):
        path = os.path.join(bench.ROOT, "profiles", name)
        if not os.path.exists(path):
            continue
        with open(path) as f:
            d = json.load(f)
        for key in ("kernel", "tokens", "sources_digest", "dram_bytes_per_launch"):
            assert key in d, (name, key)


def test_traffic_is_quoted_only_for_the_profiled_sources(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    files = bench.LAYERS_DECODE_SOURCES
    for rel in files:
        dst = root / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), dst)
    monkeypatch.setattr(bench, "ROOT", str(root))
    (root / "profiles").mkdir()
    rec = {"kernel": "k", "tokens": 1, "layers": 38, "sources_digest": bench.sources_digest(files),
           "dram_bytes_per_launch": 123.0}
    (root / "profiles" / "p.json").write_text(json.dumps(rec))
    got = bench.profiled_traffic("p.json", 1, files, 38)
    assert got == {"dram_bytes_per_launch": 123.0, "source": "profiles/p.json"}
    # another token count, another layer count, or sources edited since the capture
    assert bench.profiled_traffic("p.json", 2, files, 38) is None
    assert bench.profiled_traffic("p.json", 1, files, 4) is None
    assert bench.profiled_traffic("missing.json", 1, files) is None
    # a comment or the layout of a C/CUDA source does not change what is
    # compiled: the counters still apply; any change of code voids them
    with open(root / files[0], "a") as f:
        f.write("\n// a note\n/* and\n   another */\n\n")
    assert bench.profiled_traffic("p.json", 1, files, 38) == got
    with open(root / files[0], "a") as f:
        f.write("\nstatic int edited_since_capture;\n")
    assert bench.profiled_traffic("p.json", 1, files, 38) is None


def test_code_only_keeps_literals():
    src = 'int a = 1; // c\n/* b */ const char* s = "x // y /* z */"; char q = \'\\\'\';\n'
    assert bench.code_only(src) == 'int a = 1; const char* s = "x // y /* z */"; char q = \'\\\'\';'


def test_fp8_prefill_option(monkeypatch):
    # --fp8 selects the E4M3 prefill call for the prefill workload and, like
    # any non-default run, leaves the workloads block out; a default run
    # measures the prefill chunk with both operand types
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py", "--config", "4", "--fp8"])
    a = bench.parse()
    assert a.fp8 and a.config == 4 and not a.workloads
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert not a.fp8 and a.workloads and a.config == 1
    prefill = [w for w in bench.OTHER_WORKLOADS if w["config"] == 4]
    assert sorted(bool(w.get("fp8")) for w in prefill) == [False, True]
