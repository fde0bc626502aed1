"""The committed ncu summaries and how bench.py reads them (no GPU).

bench.py reports a kernel's measured DRAM traffic only from a summary taken
on the current kernel sources: the summary carries the sources' hash, and a
mismatch gives no figure.  Each summary also states the algorithmic bytes
per launch that its traffic is compared with; those must be the byte
model's own figure for the workload."""

import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _values(path):
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    return vals


def test_traffic_only_from_a_summary_of_the_current_sources(tmp_path, monkeypatch):
    import bench
    src = tmp_path / "kernel.cuh"
    src.write_text("// a kernel\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash(["kernel.cuh"])
    prof = tmp_path / "profiles" / "fasa_step_someworkload.md"
    prof.write_text(f"# x\n\n- kernel_source_hash: `{h}`\n- dram_bytes_per_launch: 12345\n")
    assert bench.ncu_traffic("someworkload", sources=["kernel.cuh"]) == 12345.0
    assert bench.ncu_traffic("otherworkload", sources=["kernel.cuh"]) is None  # no summary
    src.write_text("// a kernel, changed\n")  # the sources moved on: no figure
    assert bench.ncu_traffic("someworkload", sources=["kernel.cuh"]) is None
    prof.write_text(f"# x\n\n- kernel_source_hash: `{bench.kernel_source_hash(['kernel.cuh'])}`\n"
                    "- dram_bytes_per_launch: not a number\n")
    assert bench.ncu_traffic("someworkload", sources=["kernel.cuh"]) is None


@pytest.mark.parametrize("fname", sorted(f for f in os.listdir(PROFILES) if f.startswith("fasa_step_")))
def test_step_summary_states_the_byte_model(fname):
    """A step summary's algorithmic bytes are bench.py's byte model for its
    workload (full caches), and its DRAM bytes are no less than them."""
    import bench
    from workload import configs
    vals = _values(os.path.join(PROFILES, fname))
    name = re.match(r"fasa_step_(.+)\.md$", fname).group(1)
    cfg = configs.CONFIGS[name]
    model = bench.algorithmic_bytes(cfg, np.full(cfg.batch, cfg.context))
    assert int(vals["algorithmic_bytes_per_launch"]) == int(model["total"])
    assert float(vals["dram_bytes_per_launch"]) >= int(model["total"])
    assert re.fullmatch(r"[0-9a-f]{16}", vals["kernel_source_hash"])
