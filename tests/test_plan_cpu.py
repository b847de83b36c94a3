"""The decompress launch planner (csrc/zvc_plan.h) on the CPU: tests/plan_check.cpp runs it
against a model of a GB300 SM's limits, and these tests check the plans' properties: every
plan fits, the buffer is a multiple of 4 words between the minimum and the largest chunk,
several chunks share a CTA only for short chunks in launches of two waves or more, and the
cases the kernel's measurements chose it for come out as chosen."""
import json
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "activation_sparsity_compression_gb300", "csrc")
SMS = 152
CAP_MIN = 1024


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_check")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Wextra", "-Werror", "-I", CSRC,
                    os.path.join(HERE, "plan_check.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return {r["case"]: r for r in map(json.loads, out.splitlines())}


def _short(p):
    return p["mean"] * 6 <= p["full"] or p["full"] <= 1060


def test_every_plan_fits_and_is_well_formed(plans):
    for name, p in plans.items():
        if name == "occ_error":
            continue
        assert p["ok"] == 1, name
        assert p["cap"] % 4 == 0 and min(CAP_MIN, p["full"]) <= p["cap"] <= p["full"], name
        assert p["k"] in (1, 2, 4), name
        assert p["occ"] >= 1, name  # at least one CTA of the plan fits on an SM
        assert p["k"] * p["slot_bytes"] <= 232448, name


def test_several_chunks_per_cta_only_for_short_chunks_in_long_launches(plans):
    for name, p in plans.items():
        if name == "occ_error" or p["k"] == 1:
            continue
        assert _short(p), name
        assert p["chunks"] >= 2 * SMS, name


def test_cases_as_measured(plans):
    # dense data needs the largest buffer; one chunk per CTA
    for name in ("alexnet0_dense", "sweep_100", "c16384_dense", "c32768_dense"):
        assert plans[name]["cap"] == plans[name]["full"] and plans[name]["k"] == 1, name
    # 60% and 45% maps: a buffer sized from the mean, below the largest chunk
    for name in ("alexnet0_60", "alexnet1_45", "sweep_50"):
        p = plans[name]
        assert p["k"] == 1 and p["mean"] < p["cap"] < p["full"], name
        assert p["occ"] > plans["alexnet0_dense"]["occ"], name  # more chunks in flight
    # one wave (1352 chunks): the largest buffer, so no chunk is staged in pieces
    assert plans["alexnet4_20"]["cap"] == plans["alexnet4_20"]["full"]
    # sparse maps in long launches: 4 chunks per CTA, walked by one warp
    for name in ("sweep_0", "sweep_10", "c1024_sweep_50", "c32_sweep_0"):
        assert plans[name]["k"] == 4, name
    assert plans["c1024_small"]["k"] == 1  # 196 chunks: one wave
    # a batch's mean chunk leaves out the batch header and table
    assert plans["batch_25"]["k"] == 1 and plans["batch_25"]["cap"] < plans["batch_25"]["full"]


def test_degenerate_inputs(plans):
    assert plans["no_chunks"]["cap"] == plans["no_chunks"]["full"]
    assert plans["no_chunks"]["k"] == 1
    t = plans["truncated"]  # a stream smaller than its own tables: its mean is 0
    assert t["ok"] == 1 and t["mean"] == 0 and t["cap"] >= CAP_MIN
    assert plans["occ_error"]["ok"] == 0  # a failing occupancy query is reported
