"""Algorithm 1's schedule against hand-computed trajectories.

[Chelsea §三 算法流程, Algorithm 1]: B = R (n + Gamma), one round whenever
s >= B + g after prefill and after every append. Each round leaves
s' = s - floor((s - n1 - n2) / c) * m. The trajectories below were worked out
by hand for the three long-context workloads (n1=16, n2=64, c=256, g=64,
Gamma=1000).
"""
import oracle
from oracle.schedule import plan


def test_single_layer_16k():
    # B = 0.2 * 17384 = 3476.8
    assert abs(oracle.budget(16384, 0.2, 1000) - 3476.8) < 1e-9
    p = plan(16384, 0.2, 1000, 64, 16, 64, 256, r_init=0.5)
    assert [(st, s, m, s2) for st, s, _, m, s2 in p] == [
        (0, 16384, 128, 8320), (1, 8321, 128, 4225), (2, 4226, 128, 2178)]


def test_progressive_32k():
    p = plan(32768, 0.2, 1000, 64, 16, 64, 256, r_init=0.5, dr=0.05, r_min=0.1)
    assert [(st, s, m, s2) for st, s, _, m, s2 in p] == [
        (0, 32768, 128, 16512), (1, 16513, 115, 9153), (2, 9154, 102, 5584)]


def test_stack_64k():
    p = plan(65536, 0.2, 1000, 64, 16, 64, 256, r_init=0.5)
    assert [(st, s, s2) for st, s, _, _, s2 in p] == [
        (0, 65536, 32896), (1, 32897, 16513), (2, 16514, 8322)]


def test_ratio_floor_and_edges():
    assert oracle.ratio(0, 0.5, 0.05, 0.1) == 0.5
    assert oracle.ratio(20, 0.5, 0.05, 0.1) == 0.1
    assert oracle.edges_per_chunk(0.45, 256) == 115
    # 0.5 - 6*0.05 is 0.19999999999999996 in fp64; 0.2 * 256 = 51.2 -> 51 either way
    assert oracle.edges_per_chunk(oracle.ratio(6, 0.5, 0.05, 0.1), 256) == 51
    # r c integral in exact arithmetic: 0.5 - 5*0.05 = 0.25 exactly -> 64
    assert oracle.edges_per_chunk(oracle.ratio(5, 0.5, 0.05, 0.1), 256) == 64
    assert oracle.edges_per_chunk(0.5, 64) == 32
    assert not oracle.should_trigger(3540, 3476.8, 64) and oracle.should_trigger(3541, 3476.8, 64)
