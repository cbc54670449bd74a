"""CPU checks of the benchmark's roofline arithmetic (no GPU): the algorithmic bytes per launch of
the benchmark workload are 1 282 B per token-head (q, k, v, g, beta in; out) plus the fp32 final
states, and the roofline time at the measured copy bandwidth follows from them."""
import math

import pytest
import torch

import bench


def _shapes(B, T, H, init_dtype=None, nseq=None):
    """A workload dict with shapes only (meta tensors hold no memory)."""
    d = {"q": torch.empty(B, T, H, 128, dtype=torch.bfloat16, device="meta"), "cu_seqlens": None,
         "initial_state": None}
    if nseq is not None:
        d["cu_seqlens"] = torch.empty(nseq + 1, dtype=torch.int64, device="meta")
    if init_dtype is not None:
        d["initial_state"] = torch.empty(nseq or B, H, 128, 128, dtype=init_dtype, device="meta")
    return d


def test_benchmark_workload_bytes_and_roofline_time():
    nbytes, flops = bench.algorithmic(None, _shapes(8, 4096, 16))
    assert bench.BYTES_PER_TOKEN_HEAD == 1282
    assert nbytes == 1282 * 8 * 4096 * 16 + 8 * 16 * 128 * 128 * 4 == 680_525_824
    assert flops == 8 * 16 * 256 * bench.FLOPS_PER_CHUNK_HEAD
    # at the copy bandwidth measured on this hardware (6 687.8 GB/s): 101.8 us per launch
    assert nbytes / 6687.8e9 * 1e6 == pytest.approx(101.76, abs=0.01)


def test_state_bytes_count_the_initial_state_in_its_dtype():
    base, _ = bench.algorithmic(None, _shapes(1, 64, 2))
    with_bf16, _ = bench.algorithmic(None, _shapes(1, 64, 2, torch.bfloat16))
    with_fp32, _ = bench.algorithmic(None, _shapes(1, 64, 2, torch.float32))
    st = 2 * 128 * 128
    assert with_bf16 - base == 2 * st and with_fp32 - base == 4 * st


def test_varlen_states_follow_the_sequence_count():
    nbytes, flops = bench.algorithmic(None, _shapes(1, 1000, 4, torch.float32, nseq=5))
    assert nbytes == 1282 * 1000 * 4 + 5 * 4 * 128 * 128 * (4 + 4)
    assert flops == 4 * math.ceil(1000 / 16) * bench.FLOPS_PER_CHUNK_HEAD
