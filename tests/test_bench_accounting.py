"""Host-side accounting of bench.py: the algorithmic work it credits per
kernel launch, the dominant-kernel roofline, the credited flops of a stack
step, and the lookup of recorded DRAM traffic by source hash."""
import hashlib
import os

import pytest

import bench


T, D, H = 262144, 512, 1536


def test_algorithmic_work_per_kernel_family():
    # tcgen05 GEMMs and the attention projection: 2 M N K flops
    assert bench.algorithmic_work("gemm_tc_pair[16384,8192,8192]") == ("tensor", 2.0 * 16384 * 8192 * 8192)
    assert bench.algorithmic_work("attn_prep_gemm[65536,1024,512]") == ("tensor", 2.0 * 65536 * 1024 * 512)
    # the block forward: gate and down GEMMs, 4 T d h
    assert bench.algorithmic_work("block_fwd[%d,%d,%d]" % (T, D, H)) == ("tensor", 4.0 * T * D * H)
    # the backward activation kernel: only dA = dY W_down^T is credited
    assert bench.algorithmic_work("block_bwd_act[%d,%d,%d]" % (T, D, H)) == ("tensor", 2.0 * T * D * H)
    # fp32 SIMT GEMM on the CUDA cores
    assert bench.algorithmic_work("gemm_simt[128,256,784]") == ("alu", 2.0 * 128 * 256 * 784)
    # memory-bound kernels: the bytes they must move
    assert bench.algorithmic_work("sgd[17301504,0,0]") == ("hbm", 22.0 * 17301504)
    assert bench.algorithmic_work("cast[268435456,0,0]") == ("hbm", 3.0 * 268435456)
    assert bench.algorithmic_work("xent[16384,1000,0]") == ("hbm", 16384 * 1000 * 6.0 + 8.0 * 16384)
    assert bench.algorithmic_work("rmsnorm_bwd[262144,0,0]") == ("hbm", 4100.0 * 262144)
    assert bench.algorithmic_work("colsum[16384,8192,0]") == ("hbm", 2.0 * 16384 * 8192 + 4.0 * 8192)
    assert bench.algorithmic_work("mse[134217728,0,0]") == ("hbm", 6.0 * 134217728)


def test_stack_credits_the_gemms_it_runs():
    wl = bench.StackStep()
    # six 2 T d h GEMMs per block, less the first block's input gradient
    assert wl.credited_flops_per_step == (11 * 6 - 1) * 2.0 * T * D * H
    assert wl.sustained


def test_roofline_takes_the_kernel_family_with_the_most_time():
    peaks = {"hbm_gbs": 6785.5, "bf16_tflops": 1884.4, "bf16_tflops_sustained": 1692.3}
    rep = {"block_fwd[%d,%d,%d]" % (T, D, H): (11, 11 * 0.85),
           "block_bwd_act[%d,%d,%d]" % (T, D, H): (11, 11 * 0.66),
           "sgd[17301504,0,0]": (1, 0.06)}
    r = bench.roofline_entry(rep, peaks, "measured", sustained=True)
    assert r["kernel"] == "block_fwd" and r["bound"] == "tensor"
    want = 4.0 * T * D * H / 0.85e-3 / 1e12
    assert r["achieved"] == pytest.approx(want, rel=1e-6)
    assert r["peak"] == 1692.3 and r["frac"] == pytest.approx(want / 1692.3, rel=1e-4)
    assert r["share_of_kernel_time"] == pytest.approx(11 * 0.85 / (11 * 0.85 + 11 * 0.66 + 0.06),
                                                      rel=1e-3)


def test_recorded_traffic_needs_the_current_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "mlp_step_gb300" / "csrc"
    src.mkdir(parents=True)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (src / "k_block.cu").write_text("kernel source v1\n")
    sha = hashlib.sha256(b"kernel source v1\n").hexdigest()[:16]
    (prof / "block.md").write_text("traffic: block_fwd stack 497600000 %s\n"
                                   "traffic: block_fwd block 94500000 0000000000000000\n" % sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("block_fwd", "stack") == 497600000.0
    # a line captured on another source is not used
    assert bench.recorded_traffic("block_fwd", "block") is None
    # nor once the source changes
    (src / "k_block.cu").write_text("kernel source v2\n")
    assert bench.recorded_traffic("block_fwd", "stack") is None
