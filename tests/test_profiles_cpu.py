"""The committed profiler summaries (CPU only).

bench.py reads the DRAM traffic per decode launch from the summary of the
decode kernel's capture, and only while the hash recorded there matches the
kernel sources it is compiled from: a kernel edit without a new capture
turns the bench line's ``roofline.traffic`` into null.  These checks keep
the summary tied to the sources and every summary tied to the command that
made it.
"""
import glob
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_profile_matches_the_kernel_sources():
    pytest.importorskip("torch")
    import bench

    traffic = bench.traffic_from_profile()
    assert traffic is not None, (
        "profiles/paged_decode_qwen3_0p6b.txt: src_sha256 differs from the decode kernel's sources "
        f"({bench.kernel_source_sha()}); capture the kernel again")
    # one K/V pass of the workload (590,858,832 algorithmic bytes), give or take the tails' rows
    assert 590e6 <= traffic <= 1.05 * 590.9e6


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(ROOT, "profiles", "*.txt")) +
                                        glob.glob(os.path.join(ROOT, "profiles", "*.md"))))
def test_every_summary_names_its_command(path):
    with open(path) as f:
        text = f.read()
    assert "ncu " in text and "--clock-control none" in text, path
    assert "python bench.py" in text, path  # the command runs committed files only
    assert len(text) < 16384, path  # a short summary, not raw profiler output
