"""The bench's work counters and kernel label, on the CPU.

The flop count is the metric's definition (4 B H Nq Nk d, halved for a causal mask with
Nq = Nk); with key padding or a bottom-right causal mask with Nq != Nk it counts the
visible (query, key) pairs, which is checked here against the masks written out as
boolean matrices.
"""
import numpy as np
import pytest

import bench


def visible_pairs(Nq, Nk, causal, L):
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    vis = np.broadcast_to(j < min(max(L, 0), Nk), (Nq, Nk)).copy()
    if causal:
        vis &= j <= i + (Nk - Nq)
    return int(vis.sum())


@pytest.mark.parametrize("B,H,Nq,Nk,d", [(1, 2, 256, 256, 64), (2, 3, 129, 300, 128)])
def test_dense_and_half_for_causal(B, H, Nq, Nk, d):
    assert bench.algorithmic_flops(B, H, Nq, Nk, d, False) == 4.0 * B * H * Nq * Nk * d
    if Nq == Nk:
        assert bench.algorithmic_flops(B, H, Nq, Nk, d, True) == 2.0 * B * H * Nq * Nk * d


@pytest.mark.parametrize("Nq,Nk,causal,lens", [
    (128, 640, True, None),          # Nq < Nk: bottom-right causal, counted exactly
    (300, 200, True, None),          # Nq > Nk: the first rows see no key
    (256, 256, False, [256, 0]),     # padding with a fully masked batch
    (100, 400, True, [400, 37]),     # padding and a bottom-right causal mask together
])
def test_visible_pairs_against_the_masks(Nq, Nk, causal, lens):
    B, H, d = 2, 3, 64
    Ls = [Nk] * B if lens is None else lens
    want = 4.0 * H * d * sum(visible_pairs(Nq, Nk, causal, L) for L in Ls)
    got = bench.algorithmic_flops(B, H, Nq, Nk, d, causal, lens)
    if causal and Nq == Nk:  # the metric's convention: half the square
        want = 4.0 * H * d * sum(min(L, Nk) for L in Ls) * Nq / 2.0
    assert got == want


def test_row_flops_sum_to_the_total():
    Nq, Nk, d = 96, 300, 128
    for causal in (False, True):
        for L in (300, 123, 0):
            rows = sum(bench.row_flops(i, Nq, Nk, d, causal, L) for i in range(Nq))
            assert rows == 4.0 * d * visible_pairs(Nq, Nk, causal, L)


def test_kernel_label_follows_the_two_tile_rule():
    sms = 152
    # d = 64, causal: at least one pair of tiles per SM takes the two-tile kernel
    assert bench.fused_kernel_name(1, 32, 32768, 64, sms, True).startswith("attn_fwd_pair_kernel")
    assert bench.fused_kernel_name(1, 12, 2048, 64, sms, True) == "attn_fwd_kernel<64>"      # 96 pairs
    # without a causal mask, more than half the SMs' worth of pairs is enough
    assert bench.fused_kernel_name(1, 12, 2048, 64, sms, False).startswith("attn_fwd_pair_kernel")
    assert bench.fused_kernel_name(1, 9, 2048, 64, sms, False) == "attn_fwd_kernel<64>"      # 72 pairs
    assert bench.fused_kernel_name(1, 2, 256, 64, sms, False) == "attn_fwd_kernel<64>"
    assert bench.fused_kernel_name(2, 32, 8192, 128, sms, True) == "attn_fwd_kernel<128>"


def test_cpulist_parsing():
    assert bench._cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpulist("5") == {5}
    assert bench._cpulist("") == set()


def test_pages_nodes_finds_this_buffer():
    """The NUMA report reads /proc/self/maps and numa_maps: a buffer this process has
    touched must be found in some node (or the files are unavailable: None)."""
    import os
    buf = np.ones(1 << 22, dtype=np.uint8)   # 4 MiB, touched
    nodes = bench.pages_nodes(buf.ctypes.data, buf.nbytes)
    if not os.path.exists("/proc/self/numa_maps"):
        assert nodes is None
    else:
        assert nodes is None or (isinstance(nodes, dict) and all(isinstance(k, int) for k in nodes))


def test_near_gpu_restores_affinity():
    import os
    before = os.sched_getaffinity(0)
    one = {min(before)}
    with bench.near_gpu(one):
        assert os.sched_getaffinity(0) == one or len(before) == 1
    assert os.sched_getaffinity(0) == before
    with bench.near_gpu(None):          # no node information: nothing changes
        assert os.sched_getaffinity(0) == before
