"""CPU checks of bench.py's bookkeeping: the algorithmic bytes it divides by, and the rule that a recorded DRAM
traffic figure is reported only while the kernel sources it was taken on are unchanged."""
import importlib
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    sys.path.insert(0, ROOT)
    return importlib.import_module("bench")


def test_algorithmic_bytes(bench):
    from kda_linear_attention_bounded_gb300 import inputs
    # 2048 x 8 tokens x 16 heads x 1282 B + 8 x 16 initial and final states of 64 KiB
    assert bench.prefill_algorithmic_bytes(inputs.prefill_2048x8()) == 16384 * 16 * 1282 + 2 * 8 * 16 * 65536
    # 64 x 8 tokens x 16 heads x 1282 B + 64 x 16 x (1 pool read + 8 per-step states) x 64 KiB
    assert bench.verify_algorithmic_bytes(inputs.verify_64x8()) == 512 * 16 * 1282 + 64 * 16 * 9 * 65536
    step = inputs.spec_step_2048x4_64x4()
    assert bench.spec_step_algorithmic_bytes(step) == (
        8192 * 16 * 1282 + 2 * 4 * 16 * 65536 + 256 * 16 * 1282 + 64 * 16 * 5 * 65536 + 4 * (8192 + 256))


def test_traffic_record_follows_the_kernel_sources(bench, tmp_path, monkeypatch):
    # a copy of the kernel sources and a record taken on them: reported until a source changes
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    csrc = root / "kda_linear_attention_bounded_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "kda_linear_attention_bounded_gb300", "csrc"), csrc,
                    ignore=shutil.ignore_patterns("*.o", "*.so"))
    monkeypatch.setattr(bench, "ROOT", str(root))
    with open(root / "profiles" / "verify_traffic.txt", "w") as f:
        f.write(f"# a record\nsource_digest: {bench.source_digest('verify')}\ndram_bytes_per_launch: 12345\n")
    assert bench.recorded_traffic("verify") == 12345.0
    assert bench.recorded_traffic("prefill") is None        # no record
    with open(csrc / "kda_recurrent.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.recorded_traffic("verify") is None
