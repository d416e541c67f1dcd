"""Host checks of bench.py's attainable-time model of the Gram-NS product chain: its product list
follows the library's launch sequence, and its useful FLOPs add up to the pages' closed form."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import matrix_orthogonalizing_optimizer_syrk_gb300 as d3  # noqa: E402

SCHEDULES = [(5, (2, 4)), (5, ()), (5, (2,)), (3, (1, 2)), (1, ()), (8, (3, 6))]


@pytest.mark.parametrize("T,restarts", SCHEDULES)
def test_product_list_follows_the_launch_sequence(T, restarts):
    assert len(bench.gram_chain_products(1024, 4096, T, restarts)) == d3.gram_core_launch_count(T, restarts, 1024)


@pytest.mark.parametrize("T,restarts", SCHEDULES)
@pytest.mark.parametrize("k,m", [(1024, 4096), (1024, 11008), (256, 300)])
def test_useful_flops_equal_the_closed_form(T, restarts, k, m):
    """(4T + 3 alpha - 3) k^3 + r 3 (alpha - 1) k^3, the pages' FLOP count of Gram-NS with r restarts."""
    flops = sum(f for f, _ in bench.gram_chain_products(k, m, T, restarts))
    assert flops == bench.gram_flops(k, m, T, restarts)


def test_single_iteration_bytes():
    """T = 1: X X^T, the polynomial, the fused W update; 16-bit iterates, fp32 W."""
    k, m = 256, 1000
    seq = bench.gram_chain_products(k, m, 1, ())
    assert [b for _, b in seq] == [2 * (k * m + k * k), 2 * 2 * k * k, 2 * (k * k + k * m) + 8 * k * m]


def test_bound_is_the_slower_of_tensor_and_hbm_per_product():
    k, m = 1024, 4096
    fast_hbm = bench.gram_chain_bound_ms([(1, 4096, m)], 1000.0, 1e12)
    flops = sum(f for f, _ in bench.gram_chain_products(k, m))
    assert fast_hbm == pytest.approx(flops / 1e15 * 1e3)
    fast_tc = bench.gram_chain_bound_ms([(1, 4096, m)], 1e12, 1000.0)
    nbytes = sum(b for _, b in bench.gram_chain_products(k, m))
    assert fast_tc == pytest.approx(nbytes / 1e12 * 1e3)


def test_carried_step_passes_the_previous_selection():
    """The timed loop's step: the first call carries nothing in, every later call carries the
    previous call's rows (the same buffer it writes) with mu, and every call defers its own decay."""
    calls = []

    class FakeLib:
        @staticmethod
        def step(W, M, G, **kw):
            calls.append(kw)

    x = {"W": "W", "M": "M", "Gs": ["G0", "G1"], "sel": "sel"}
    for s in range(3):
        bench.carried_step(FakeLib, x, s % 2, "ws", "status")
    assert calls[0]["carry"] is None
    assert all(c["carry"] == ("sel", bench.MU) for c in calls[1:])
    assert all(c["defer"] is True and c["sel_out"] == "sel" for c in calls)


def test_roofline_peak_follows_the_clock_record():
    """The burst bf16 figure was measured at the maximum SM clock: it is the denominator when the
    run's median clock sat within 3% of the maximum; otherwise (or without a clock record) the
    sustained one is."""
    assert bench.clock_at_max({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})
    assert bench.clock_at_max({"sm_mhz": 2010.0, "sm_max_mhz": 2070.0})
    assert not bench.clock_at_max({"sm_mhz": 1995.0, "sm_max_mhz": 2070.0})
    assert not bench.clock_at_max({"sm_mhz": 1515.0, "sm_max_mhz": 2070.0})
    assert not bench.clock_at_max({"error": "nvidia-smi unavailable"})
    assert not bench.clock_at_max(None)


@pytest.mark.parametrize("B,expect", [(128, [0, 64, 127]), (96, [0, 48, 95]), (2, [0, 1]), (1, [0])])
def test_oracle_sample_is_first_middle_last(B, expect):
    assert bench.sample_indices(B) == expect


def test_recorded_traffic_is_keyed_to_the_kernel_source():
    """traffic.json holds a per-launch byte count for the GEMM family, valid only for the source it
    was measured on: the bench reports it when the hash matches, null for an unknown kernel."""
    v = bench.recorded_traffic("tc_gemm_kernel (all tcgen05 GEMM launches of the Gram-NS chain)")
    assert v is None or 1e9 < v < 3e9
    assert bench.recorded_traffic("no such kernel") is None
