"""Recorded-plan table of sgemm_f32_autotune on the host side (no GPU): loading, saving,
clearing, and the planner using a recorded plan for exactly its key."""
import os

import pytest

import dense_fp32_matrix_08_gb300 as sg


@pytest.fixture(autouse=True)
def _empty_table():
    sg.sgemm_f32_tune_clear()
    yield
    sg.sgemm_f32_tune_clear()


# flags of a row-major problem with 16-byte aligned A, B and lda, ldb multiples of 4
# (TMA-able = 4, K-paired-able = 8, A and B TMA-addressable = 64, 128) and beta != 0 (32)
FLAGS_ALIGNED_BETA = 4 | 8 | 32 | 64 | 128


def test_load_applies_to_its_key_only(tmp_path):
    f = tmp_path / "t.txt"
    f.write_text(f"# comment\n152 1000 1000 1000 {FLAGS_ALIGNED_BETA} 2 3 0.5\n")
    assert sg.sgemm_f32_tune_load(f) == 1
    assert sg.sgemm_f32_tune_count() == 1
    p = sg.sgemm_f32_plan(1000, 1000, 1000, 1000, 1000, 1000, 1.0, 1.0, 152)
    assert (p["variant"], p["split"]) == (2, 3)
    # another key: beta == 0, another SM count, another shape, another alignment class
    for args in [(1000, 1000, 1000, 1000, 1000, 1000, 1.0, 0.0, 152),
                 (1000, 1000, 1000, 1000, 1000, 1000, 1.0, 1.0, 148),
                 (1000, 1000, 999, 999, 1000, 1000, 1.0, 1.0, 152),
                 (1000, 1000, 1000, 1001, 1000, 1000, 1.0, 1.0, 152)]:
        assert sg.sgemm_f32_plan(*args)["variant"] != 2 or \
            sg.sgemm_f32_plan(*args)["split"] != 3


def test_save_load_round_trip(tmp_path):
    src = tmp_path / "a.txt"
    src.write_text(f"152 512 640 768 {FLAGS_ALIGNED_BETA} 30 -1 1.25\n"
                   f"152 100 200 300 {FLAGS_ALIGNED_BETA} 16 1 0.125\n")
    assert sg.sgemm_f32_tune_load(src) == 2
    out = tmp_path / "b.txt"
    assert sg.sgemm_f32_tune_save(out) == 2
    lines = [ln for ln in out.read_text().splitlines() if not ln.startswith("#")]
    assert sorted(lines) == sorted([f"152 512 640 768 {FLAGS_ALIGNED_BETA} 30 -1 1.250000",
                                    f"152 100 200 300 {FLAGS_ALIGNED_BETA} 16 1 0.125000"])
    sg.sgemm_f32_tune_clear()
    assert sg.sgemm_f32_tune_count() == 0
    assert sg.sgemm_f32_tune_load(out) == 2
    assert sg.sgemm_f32_plan(512, 640, 768, 768, 640, 640, 1.0, 2.0, 152)["variant"] == 30


def test_same_key_replaces(tmp_path):
    f = tmp_path / "t.txt"
    f.write_text(f"152 64 64 64 {FLAGS_ALIGNED_BETA} 2 1 1.0\n"
                 f"152 64 64 64 {FLAGS_ALIGNED_BETA} 16 1 0.5\n")
    assert sg.sgemm_f32_tune_load(f) == 2
    assert sg.sgemm_f32_tune_count() == 1
    assert sg.sgemm_f32_plan(64, 64, 64, 64, 64, 64, 1.0, 1.0, 152)["variant"] == 16


def test_bad_lines_and_paths(tmp_path):
    n = sg.sgemm_f32_num_variants()
    f = tmp_path / "t.txt"
    f.write_text(f"152 64 64 64 {FLAGS_ALIGNED_BETA} {n} 1 1.0\n"   # variant out of range
                 "152 64 64\n"                                       # too few fields
                 f"0 64 64 64 {FLAGS_ALIGNED_BETA} 2 1 1.0\n"        # no SMs
                 f"152 64 64 64 {FLAGS_ALIGNED_BETA} 2 1 1.0\n")     # valid
    assert sg.sgemm_f32_tune_load(f) == -3
    assert sg.sgemm_f32_tune_count() == 1
    assert sg.sgemm_f32_tune_load(tmp_path / "missing.txt") == -2
    assert sg.lib.sgemm_f32_tune_load(None) == -1
    assert sg.lib.sgemm_f32_tune_save(None) == -1
    assert sg.sgemm_f32_tune_save(os.path.join(tmp_path, "no", "such", "dir.txt")) == -2


def test_env_force_switch():
    """SGEMM_F32_FORCE pins the automatic plan of every entry point to a configuration (a
    benchmarking switch), except where that configuration cannot run the problem."""
    import subprocess
    import sys
    code = ("import dense_fp32_matrix_08_gb300 as sg\n"
            "p = sg.sgemm_f32_plan(4096, 4096, 4096, 4096, 4096, 4096, 1.0, 1.0, 152)\n"
            "q = sg.sgemm_f32_plan(64, 64, 64, 64, 64, 64, 1.0, 1.0, 152)\n"
            "print(p['variant'], p['split'], q['variant'])\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, SGEMM_F32_FORCE="16:1")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                         text=True, check=True).stdout.split()
    assert out[:2] == ["16", "1"] and out[2] == "16"
    # an out-of-range configuration is ignored: the automatic plans stay as they are
    env = dict(os.environ, SGEMM_F32_FORCE="999")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                         text=True, check=True).stdout.split()
    plain = subprocess.run([sys.executable, "-c", code], cwd=root,
                           env={k: v for k, v in os.environ.items() if k != "SGEMM_F32_FORCE"},
                           capture_output=True, text=True, check=True).stdout.split()
    assert out == plain
