"""Pins of the oracle's memory and communication accounting against the
figures the pages print (golden fixtures) and the closed forms of a second
page (the oracle was written from the itwiki stage table; the Hinglish notes
state the same result as separate formulas)."""
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_stage_table_7p5b_64_gpus():
    # "ZeRO (딥 러닝)", ZeRO-DP의 세 단계: 120 / 31.4 / 16.6 / 1.9 GB and 2/2/2/3 psi
    rows = list(_rows("model_states_7p5b_64.txt"))
    assert len(rows) == 4
    for stage, gb, comm in rows:
        total = oracle.model_state_bytes(7.5e9, 64, int(stage))[3] / 1e9
        assert round(total, 1) == float(gb)
        assert oracle.comm_volume(int(stage)) == float(comm)


def test_stage_table_exact_values():
    # the unrounded values behind the printed ones: (16, 4+12/64, 2+14/64, 16/64) * 7.5
    exact = [120.0, 31.40625, 16.640625, 1.875]
    for stage, want in enumerate(exact):
        assert oracle.model_state_bytes(7.5e9, 64, stage)[3] / 1e9 == pytest.approx(want, rel=1e-15)


def test_worked_examples():
    g = {r[0]: float(r[1]) for r in _rows("memory_examples.txt")}
    # 16 bytes per parameter under standard DP (stage 0)
    assert oracle.model_state_bytes(1.3e9, 8, 0)[3] / 1e9 == pytest.approx(g["dp_1p3b_gb"])
    assert oracle.model_state_bytes(1.3e9, 8, 3)[3] / 1e9 == pytest.approx(g["zero3_1p3b_8_gb"])
    p, gr, o, tot = oracle.model_state_bytes(1.5e9, 1, 0)
    assert tot / 1e9 == pytest.approx(g["gpt2_1p5b_states_gb"])
    assert p / 1e9 == pytest.approx(g["gpt2_1p5b_fp16_weights_gb"])
    # the optimizer term alone: fp32 master (4) of 175B -> 700 GB; K=12 -> 2.1 TB
    assert oracle.model_state_bytes(175e9, 1, 0, k=4.0)[2] / 1e9 == pytest.approx(g["gpt3_fp32_weights_gb"])
    assert oracle.model_state_bytes(175e9, 1, 0)[2] / 1e12 == pytest.approx(g["gpt3_adam_state_tb"])
    per_gpu = 530e9 / (8 * 35)
    assert round(per_gpu / 1e9, 1) == g["mtnlg_params_per_gpu_b"]
    assert round(oracle.model_state_bytes(per_gpu, 1, 0, k=4.0)[2] / 1e9, 1) == g["mtnlg_fp32_gb"]


@pytest.mark.parametrize("psi", [1.0, 7.5e9, 1.3e9, 123456789.0])
@pytest.mark.parametrize("n", [1, 2, 8, 64, 1000])
def test_closed_forms_of_the_hinglish_notes(psi, n):
    # "Data parallelism and ZeRO optimization": M_ZeRO-1 = 4 psi + 12 psi / N,
    # M_ZeRO-2 = 2 psi + 14 psi / N, M_ZeRO-3 = 16 psi / N, standard DP 16 psi.
    want = [16 * psi, 4 * psi + 12 * psi / n, 2 * psi + 14 * psi / n, 16 * psi / n]
    for stage in range(4):
        assert oracle.model_state_bytes(psi, n, stage)[3] == pytest.approx(want[stage], rel=1e-14)


def test_large_n_reduction_factors():
    # "ZeRO (딥 러닝)": for large N_d stage 1 saves about 4x, stage 2 about 8x,
    # stage 3 in proportion to the GPU count (64x with 64 GPUs).
    psi, n = 1e9, 1e9
    base = oracle.model_state_bytes(psi, n, 0)[3]
    assert base / oracle.model_state_bytes(psi, n, 1)[3] == pytest.approx(4.0, rel=1e-6)
    assert base / oracle.model_state_bytes(psi, n, 2)[3] == pytest.approx(8.0, rel=1e-6)
    assert base / oracle.model_state_bytes(psi, 64, 3)[3] == pytest.approx(64.0, rel=1e-15)


def test_stage3_comm_is_one_and_a_half_times_dp():
    # "ZeRO (딥 러닝)", 왜 통신량이 늘지 않는가: 3 psi against 2 psi (1.5x)
    assert oracle.comm_volume(3) / oracle.comm_volume(0) == 1.5
