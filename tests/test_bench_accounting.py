"""The benchmark's algorithmic bytes per parameter (the numerator of every
roofline fraction it reports) against the closed forms of the method's
minimum HBM traffic, workload by workload."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_headline_clipped_step():
    # reduce pass 2N_d + 4 (fp32 reduced gradient written), Adam pass 30
    w = bench.workload(2)
    assert (w["psi"], w["n_d"], w["clip"]) == (124_439_808, 8, 1.0)
    assert w["bytes_per_param"] == (2 * 8 + 4) + 30 == 50


@pytest.mark.parametrize("cfg,n_d,want", [(1, 4, 2 * 4 + 26), (3, 8, 2 * 8 + 26)])
def test_fused_step(cfg, n_d, want):
    w = bench.workload(cfg)
    assert w["n_d"] == n_d and w["bytes_per_param"] == want


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 64])
def test_sweep_and_quantized_variants(n_d):
    assert bench.workload(5, nd=n_d)["bytes_per_param"] == 2 * n_d + 26
    # int8 gather: codes (1) + dequantized bf16 (2) instead of the plain param (2), one scale per 2048
    assert bench.workload(5, nd=n_d, qgather=True)["bytes_per_param"] == 2 * n_d + 27 + 4.0 / 2048
    # qgZ receiver: one int8 code and one fp32 scale per 2048 per rank
    assert bench.workload(5, nd=n_d, qgz=True)["bytes_per_param"] == n_d * (1 + 4.0 / 2048) + 26


@pytest.mark.parametrize("gathers", [1, 2])
def test_zero3_layer(gathers):
    w = bench.workload(4, gathers=gathers)
    assert w["layers"] == 8 and w["psi"] == 218_112_000
    # each gather reads a 16-bit shard and writes the gathered layer
    assert w["bytes_per_param"] == 2 * 16 + 26 + 4 * gathers
    assert w["psi_total"] == 8 * 218_112_000
    # with block-int8 gathers (qwZ): the shard read, codes + scales + dequantized bf16 written
    q = bench.workload(4, gathers=gathers, qgather=True)
    assert q["bytes_per_param"] == 2 * 16 + 26 + (5 + 4.0 / 2048) * gathers
    assert q["name"].endswith("_qgather") and q["stage"] == 3


@pytest.mark.parametrize("k", [2, 4, 8])
def test_accumulation(k):
    # micro-batch 1 writes the fp32 accumulator, 2..k-1 read and write it,
    # the clipped step at micro-batch k reads it in its reduce pass
    w = bench.workload(2, accum=k)
    n = w["n_d"]
    assert w["bytes_per_param"] == (2 * n + 4) + (k - 2) * (2 * n + 8) + (2 * n + 38)
    assert w["bytes_per_param"] == 2 * n * k + 8 * (k - 1) + 34
    w1 = bench.workload(1, accum=k)
    assert w1["bytes_per_param"] == 2 * 4 * k + 8 * (k - 1) + 26


@pytest.mark.parametrize("cfg,n_d,clip", [(2, 8, True), (1, 4, False)])
def test_quantized_variants_of_the_other_zero2_workloads(cfg, n_d, clip):
    q = n_d * (1 + 4.0 / 2048)
    # clipped qgZ with n_d > 4: reduce pass over codes + scales writing the fp32
    # reduced gradient (4), then the Adam pass (30)
    assert bench.workload(cfg, qgz=True)["bytes_per_param"] == (q + 34 if clip else q + 26)
    # clipped int8 gather with n_d > 4: the reduce pass writes the fp32
    # reduced gradient (2 n_d + 4), the Adam pass with the int8 gather reads it
    # with the state and writes state, codes and dequantized bf16 (4 + 24 + 3)
    want = (2 * n_d + 4) + (4 + 27 + 4.0 / 2048) if clip else 2 * n_d + 27 + 4.0 / 2048
    assert bench.workload(cfg, qgather=True)["bytes_per_param"] == want
    # n_d <= 4: a read-only reduce pass (2 n_d) before the fused step
    assert bench.workload(5, nd=4, qgather=True)["bytes_per_param"] == 2 * 4 + 27 + 4.0 / 2048


def test_quantized_variant_names():
    # the names key the stored ncu traffic of the N_d sweep
    assert bench.workload(5, nd=2, qgather=True)["name"] == "zero2_psi2p28_nd2_qgather"
    assert bench.workload(5, nd=8, qgz=True)["name"] == "zero2_psi2p28_nd8_qgz"
    assert bench.workload(2, qgz=True)["name"] == "zero2_gpt2small_psi124439808_nd8_adamw_clip1_qgz"


@pytest.mark.parametrize("cfg,n_d,clip", [(5, 8, False), (2, 8, True)])
def test_both_quantized_exchanges(cfg, n_d, clip):
    # int8 codes + scales in, int8 codes + scale + dequantized bf16 out; clipped
    # (n_d > 4), a reduce pass over the codes writing the fp32 reduced gradient
    # first, which the Adam pass with the int8 gather reads
    q = n_d * (1 + 4.0 / 2048)
    w = bench.workload(cfg, qgz=True, qgather=True)
    assert w["bytes_per_param"] == ((q + 4) + (4 + 27 + 4.0 / 2048) if clip else q + 27 + 4.0 / 2048)
    assert w["name"].endswith("_qgz_qgather") and w["pad"] == 16


def test_variants_that_do_not_apply_are_refused():
    for cfg, kw in ((3, dict(qgz=True)), (4, dict(qgz=True)), (4, dict(qgz=True, qgather=True)),
                    (4, dict(qgather=True, param_dtype="fp16"))):
        with pytest.raises(SystemExit):
            bench.workload(cfg, **kw)
    with pytest.raises(SystemExit):
        bench.workload(4, accum=2)
    with pytest.raises(SystemExit):
        bench.workload(2, serial=True)
    with pytest.raises(SystemExit):
        bench.workload(4, stage=2)
    with pytest.raises(SystemExit):
        bench.workload(5, qgather=True, param_dtype="fp16")


def test_default_workload_is_the_largest_single_gpu_one():
    # the ZeRO-3 layer loop over 8 Llama-3-8B-shaped layers, gathers on a second stream
    args = bench.build_parser().parse_args([])
    w = bench.workload_from_args(args)
    assert w["name"] == "zero3_llama3_8b_8layers_psil218112000_nd16" and w["overlap"]
    assert w["psi_total"] == 8 * 218_112_000 == 1_744_896_000
    assert w["psi_total"] * w["bytes_per_param"] == pytest.approx(108.18e9, rel=1e-3)
    # the largest workload by bytes per step
    for cfg in (1, 2, 3, 5):
        o = bench.workload(cfg)
        assert o["psi_total"] * o["bytes_per_param"] < w["psi_total"] * w["bytes_per_param"]


def test_both_arms_print_the_same_config():
    for argv in ([], ["--config", "3", "--param-dtype", "fp16", "--stage", "1"], ["--config", "2"]):
        w = bench.workload_from_args(bench.build_parser().parse_args(argv))
        assert bench.config_of(w, 1) == bench.config_of(bench.workload_from_args(
            bench.build_parser().parse_args(argv + ["--impl", "reference"])), 1)


def test_fp16_parameter_and_stage_labels():
    w = bench.workload(3, param_dtype="fp16", stage=1)
    assert w["name"] == "zero1_gpt2xl_psi1500000000_nd8_fp16_lossscale_params_fp16"
    assert w["stage"] == 1 and w["pdt"] == "fp16" and w["bytes_per_param"] == 2 * 8 + 26
    assert bench.config_of(w, 1)["param_dtype"] == "fp16"
    assert bench.workload(3)["pdt"] == "bf16"


def test_kernel_source_hash_ignores_comments_and_layout():
    # the traffic table is keyed on the engine's code: a comment or a
    # re-indented line leaves the key as it was, a changed token does not
    code = "int a = 1; // one\n/* two\n three */  float b  =\n 2.0f;"
    assert bench._code_only(code) == "int a = 1; float b = 2.0f;"
    assert bench._code_only(code.replace("// one", "// uno")) == bench._code_only(code)
    assert bench._code_only(code.replace("2.0f", "3.0f")) != bench._code_only(code)
    assert len(bench.kernel_source_hash()) == 12
