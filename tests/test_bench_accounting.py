"""bench.py's roofline accounting on the host: the algorithmic work of the
scope table (per token and head 12 d^2 + 8 C d + 4 C d + C^2/3 FLOP; q, k,
v, o, gates and states as HBM bytes), with the prepared blocks kept out of
the algorithmic bytes."""
import pytest

import bench
import workloads as W


def test_path_flops_per_token_head():
    assert bench.path_flops_per_token_head(128) == 12 * 128 * 128 + 12 * 64 * 128 + 64 * 64 // 3
    assert bench.path_flops_per_token_head(128) == 296277


def test_prefill_400m_bytes_and_flops():
    x = W.make_prefill(W.PREFILL_400M)
    by, fl = bench.algorithmic(x, "call")
    th = 8 * 2048 * 8
    state = 64 * 128 * 128 * 4
    assert by == th * (4 * 128 * 2 + 3 * 4) + 2 * state + 2 * state   # zero S0, M0 are read
    assert by == 152567808
    assert fl == th * 296277
    sb, sf = bench.algorithmic(x, "state")
    assert sb == th * 4 * 128 * 2 + 4 * state
    assert sf == th * (12 * 128 * 128 + 4 * 64 * 128)
    pb, _ = bench.algorithmic(x, "prep")
    assert pb == th * (2 * 128 * 2 + 3 * 4)
    # the intermediate is reported beside, never inside, the algorithmic bytes
    assert bench.intermediate_bytes(x, True) == 18432 * (8 * 32) * 8


def test_varlen_has_no_initial_state_reads():
    x = W.make_prefill(W.VARLEN_PACKED)
    b = bench.io_bytes(x)
    assert b["states_in"] == 0
    assert b["states_out"] == 2 * x["n_seq"] * 16 * 128 * 128 * 4
    assert sum(bench.seq_lengths(x)) == 32768


def test_roofline_binding_side():
    x = W.make_prefill(W.PREFILL_400M)
    peaks = {"hbm_gbs": 6785.2, "bf16_tflops": 1904.9}
    r = bench.roofline_of(x, "call", True, 0.1, peaks, "measured")
    by, fl = bench.algorithmic(x, "call")
    # 152.6 MB at 6.79 TB/s (22.5 us) binds over 38.8 GFLOP at 1.9 PFLOP/s (20.4 us)
    assert r["bound"] == "hbm"
    assert r["frac"] == pytest.approx(by / 1e-4 / 1e9 / 6785.2)
    assert r["other_roof_frac"] == pytest.approx(fl / 1e-4 / 1e12 / 1904.9)


def test_fp32_state_pass_peak_is_a_third_of_bf16():
    w = W.Workload("acc_fp32", B=1, T=2048, H=2, D=128, dtype="fp32", state="none", seed=0)
    x = W.make_prefill(w)
    peaks = {"hbm_gbs": 6785.2, "bf16_tflops": 1904.9}
    r = bench.roofline_of(x, "state", True, 1e-9, peaks, "measured")   # FLOP-bound at d = 128
    assert r["bound"] == "tensor" and r["peak"] == pytest.approx(1904.9 / 3)
    p = bench.roofline_of(x, "prep", True, 1e-9, peaks, "measured")
    assert p["bound"] == "alu"                      # the fp32 prep's inverse: CUDA cores
    # fp32 intermediates: the split prepared blocks and the q, k, v parts
    assert bench.intermediate_bytes(x) == 34816 * 32 * 2 + 2 * 3 * 2 * 2048 * 2 * 128


def test_backward_bytes_varlen():
    # q, k, v, dO in and dq, dk, dv out (bf16), four gates in and four
    # gradients out (fp32), every chunk's entry states (bf16, as saved), and per
    # (sequence, head) the final-state adjoints in and dS0, dM0 out
    x = W.make_prefill(W.VARLEN_PACKED)
    lens = bench.seq_lengths(x)
    th = 32768 * 16
    chunks = sum((n + 63) // 64 for n in lens) * 16
    assert chunks == 523 * 16
    want = th * (7 * 128 * 2 + 8 * 4) + chunks * 2 * 128 * 128 * 2 + len(lens) * 16 * 4 * 128 * 128 * 4
    assert bench.bwd_bytes(x) == want


def test_backward_flops_per_token_head():
    # the vector-Jacobian product's state products (24 d^2 in the chunk
    # products, 12 d^2 in the reverse chain), 14 C d chunk-local, C^2 / 3
    assert bench.bwd_flops_per_token_head(128) == 36 * 128 * 128 + 14 * 64 * 128 + 64 * 64 // 3
