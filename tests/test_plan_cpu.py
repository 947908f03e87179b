"""The tensor-core kernel's work plan, checked on the host (no GPU): the plan header is plain
integer arithmetic, compiled here with g++ and run over many problem sizes and grid sizes."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
def test_plan_covers_every_tile_once_and_every_look_back_resolves(tmp_path):
    exe = str(tmp_path / "plan_check")
    src = os.path.join(ROOT, "tests", "plan_check.cpp")
    subprocess.run(["g++", "-std=c++17", "-O2", "-Wall", "-o", exe, src], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 violations" in r.stdout


MUTANTS = {
    # a range's last tile dropped
    "k1_off_by_one": ("pl.k1 = (int)((end - 1) % T + 1);", "pl.k1 = (int)((end - 1) % T);"),
    # a middle piece taken for a tail piece
    "middle_misread": ("if (pl.u0 == pl.u1 && pl.k0 > 0 && pl.k1 < T) {",
                       "if (pl.u0 == pl.u1 && pl.k0 > 0 && pl.k1 < T - 1) {"),
    # a head piece that publishes nothing
    "head_unpublished": ("return Item{pl.u1, 0, pl.k1, 0, kInitH0, pl.p1 ? kFinNone : kFinIncl};",
                         "return Item{pl.u1, 0, pl.k1, 0, kInitH0, kFinNone};"),
    # mode 2 keeping the head's state-only item that the separate kernel runs
    "mode2_keeps_state_only_item": ("pl.n_pre = head ? 1 + (kExt ? 0 : pl.p1) : 0;",
                                    "pl.n_pre = head ? 1 + pl.p1 : 0;"),
    # the tail piece starting from the initial state instead of looking back
    "tail_no_look_back": ("return Item{pl.u0, pl.k0, (pl.u0 == pl.u1) ? pl.k1 : T, 0, kInitLookback, kFinFinal};",
                          "return Item{pl.u0, pl.k0, (pl.u0 == pl.u1) ? pl.k1 : T, 0, kInitH0, kFinFinal};"),
    # the look-back rule taking an aggregate also from the head piece's CTA
    # segments taken half as long as they may be (more records than the workspace holds)
    "segments_overflow": ("const int64_t zr = (2 * t1) / recs + ((2 * t1) % recs != 0);",
                          "const int64_t zr = t1 / recs + (t1 % recs != 0);"),
    # the next piece's segments starting one grid index too early (two CTAs on one segment)
    "segments_index": ("        s += pieces[q].nseg;", "        s += pieces[q].nseg - (pieces[q].nseg > 1);"),
    "lookback_rule": ("return pass1_mode != 0 && (int64_t)jp * total / n_ctas > (int64_t)u * n_tiles;",
                      "return pass1_mode != 0 && (int64_t)jp * total / n_ctas >= (int64_t)u * n_tiles;"),
}


@pytest.mark.skipif(shutil.which("g++") is None, reason="no host C++ compiler")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_plan_check_catches_a_planted_mistake(tmp_path, name):
    old, new = MUTANTS[name]
    hdr = open(os.path.join(ROOT, "mamba_ssd_scan_05_b300", "csrc", "tc_plan.cuh")).read()
    assert hdr.count(old) == 1, "mutation anchor not found"
    (tmp_path / "tc_plan.cuh").write_text(hdr.replace(old, new))
    src = open(os.path.join(ROOT, "tests", "plan_check.cpp")).read().replace(
        '"../mamba_ssd_scan_05_b300/csrc/tc_plan.cuh"', '"tc_plan.cuh"')
    (tmp_path / "plan_check.cpp").write_text(src)
    exe = str(tmp_path / "plan_check")
    subprocess.run(["g++", "-std=c++17", "-O2", "-o", exe, str(tmp_path / "plan_check.cpp")],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "FAIL" in r.stdout, f"mutant {name} not caught"
