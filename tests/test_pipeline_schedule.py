"""Barrier schedules of the grouped-GEMM kernels, checked on the host.

tests/pipeline_schedule_check.cpp is compiled against the schedule functions the CUDA
kernels call (nvfp4_mixture_experts_stage_gb300/csrc/pipeline.cuh) and enumerates, for
many ring sizes, k-block counts and tile counts, which use of which barrier every
waiter waits for.  An mbarrier wait tests only the parity of a phase, so each waiter
must see the uses of each of its barriers in order, none skipped.  The kernels'
earlier schedules (two copiers alternating on one scale barrier per ring entry; two
streaming issuers for an odd k-block count) must be flagged, so the check is known to
catch the mistake it guards against."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def report(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("sched") / "pipeline_schedule_check")
    subprocess.run([cxx, "-std=c++17", "-O1", "-o", exe, os.path.join(HERE, "pipeline_schedule_check.cpp")],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return {line.split()[1]: int(line.split()[2]) for line in out.splitlines() if line.startswith("violations")}


def test_current_schedules_never_skip_a_phase(report):
    assert report["pair"] == 0
    assert report["stream"] == 0


def test_producer_teardown_phase_from_the_stage_count(report):
    """The producers keep a count of issued stages, not a record per ring entry; the
    parity of each entry's last use follows from the count."""
    assert report["ring_teardown"] == 0
    assert report["ring_teardown_naive"] > 0


def test_earlier_schedules_are_flagged(report):
    assert report["pair_shared_barrier"] > 0
    assert report["stream_always_two_odd"] > 0
    # for an even k-block count two issuers were always safe
    assert report["stream_always_two_even"] == 0
