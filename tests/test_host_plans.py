"""Host logic of the work partitions, checked in the library's own host code
(the same functions the kernels evaluate on the device) through C-ABI
self-checks that need no GPU:
* the split-KV decode (rf_selftest_decode_plan): the partition of the
  sequences' keys into pieces, the CTA that takes each piece, the workspace
  slot of each partial state and the order in which the merge reads them;
* the FP8 GEMM (rf_selftest_fp8_schedule): the tiles of the output, whole
  and in column halves, over the CTA pairs;
* the MoE gate (rf_selftest_moe_plan): the cluster split of D and the token
  tiles chosen by the host's cost model."""
import random

import pytest

import __graft_entry__

_build = __graft_entry__._load_build_module()


@pytest.fixture(scope="module")
def rf():
    _build.build()
    import cascaded_reductions_loop_gb300 as m
    return m


@pytest.mark.parametrize("B,Hkv,Lk", [(32, 8, 2048), (32, 8, 32768), (64, 1, 4096), (1, 1, 1),
                                      (1, 1, 31), (1, 1, 33), (3, 5, 1000), (7, 3, 65)])
@pytest.mark.parametrize("sms", [1, 2, 7, 148, 152, 1000])
def test_automatic_partition(rf, B, Hkv, Lk, sms):
    assert rf.rf_selftest_decode_plan(B, Hkv, Lk, 0, sms) == 0


@pytest.mark.parametrize("B,Hkv,Lk", [(32, 8, 2048), (2, 3, 100), (1, 1, 1), (5, 1, 37)])
@pytest.mark.parametrize("S", [1, 2, 3, 8, 16, 31])
@pytest.mark.parametrize("sms", [1, 5, 152])
def test_explicit_segments(rf, B, Hkv, Lk, S, sms):
    if S > Lk:
        assert rf.rf_selftest_decode_plan(B, Hkv, Lk, S, sms) == -1
    else:
        assert rf.rf_selftest_decode_plan(B, Hkv, Lk, S, sms) == 0


def test_every_segment_count_of_a_short_sequence(rf):
    for Lk in (1, 2, 3, 31, 32, 33, 64, 95):
        for S in range(1, Lk + 1):
            for sms in (1, 3, 152):
                assert rf.rf_selftest_decode_plan(2, 3, Lk, S, sms) == 0, (Lk, S, sms)


def test_random_shapes(rf):
    rng = random.Random(12345)
    for _ in range(3000):
        B, Hkv = rng.randint(1, 40), rng.choice([1, 2, 4, 8, 16])
        Lk = rng.choice([rng.randint(1, 64), rng.randint(1, 5000), rng.randint(1, 70000)])
        sms = rng.choice([1, 2, 3, 64, 132, 148, 152, rng.randint(1, 400)])
        S = 0 if rng.random() < 0.7 else rng.randint(1, min(Lk, 40))
        assert rf.rf_selftest_decode_plan(B, Hkv, Lk, S, sms) == 0, (B, Hkv, Lk, S, sms)


def test_largest_shapes(rf):
    # B * Hkv * Lk just below 2^31, the limit the call accepts
    assert rf.rf_selftest_decode_plan(64, 64, 524287, 0, 152) == 0
    assert rf.rf_selftest_decode_plan(1, 1, 2 ** 31 - 1, 0, 152) == 0
    assert rf.rf_selftest_decode_plan(4, 8, 65536, 64, 152) == 0


def test_refused_shapes(rf):
    for args in [(0, 1, 1, 0, 1), (1, 0, 1, 0, 1), (1, 1, 0, 0, 1), (1, 1, 10, 11, 1),
                 (1, 1, 10, -1, 1), (1, 1, 10, 0, 0), (64, 64, 524288, 0, 152),
                 (1 << 20, 1 << 20, 0, 0, 152), (1 << 16, 1 << 16, 1, 0, 152)]:
        assert rf.rf_selftest_decode_plan(*args) == -1, args


# ------------------------------------------------ FP8 GEMM tile schedule


@pytest.mark.parametrize("clusters", [1, 2, 3, 7, 64, 74, 76])
@pytest.mark.parametrize("M,N", [(4096, 4096), (1, 1), (256, 256), (257, 255), (4096, 128),
                                 (100, 4096), (5000, 3000), (33, 8000)])
def test_fp8_schedule(rf, M, N, clusters):
    assert rf.rf_selftest_fp8_schedule(M, N, clusters) == 0


def test_fp8_schedule_random_shapes(rf):
    rng = random.Random(777)
    for _ in range(2000):
        M, N = rng.randint(1, 9000), rng.randint(1, 9000)
        clusters = rng.choice([1, 2, 3, 5, 64, 66, 74, 76, rng.randint(1, 300)])
        assert rf.rf_selftest_fp8_schedule(M, N, clusters) == 0, (M, N, clusters)


def test_fp8_schedule_refused(rf):
    for args in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (1, 1, 4097), (1 << 20, 1 << 20, 76)]:
        assert rf.rf_selftest_fp8_schedule(*args) == -1, args


# ------------------------------------------------------ MoE gate tile plan


@pytest.mark.parametrize("E", [1, 8, 32, 64, 100, 128, 192, 256])
@pytest.mark.parametrize("T,D", [(8192, 4096), (1, 8), (7, 64), (1000, 128), (65536, 1024),
                                 (65535 * 120, 4096)])
@pytest.mark.parametrize("sms", [1, 2, 148, 152, 1000])
def test_moe_plan(rf, T, D, E, sms):
    assert rf.rf_selftest_moe_plan(T, D, E, sms) == 0


def test_moe_plan_random_shapes(rf):
    rng = random.Random(4242)
    for _ in range(3000):
        T = rng.choice([rng.randint(1, 300), rng.randint(1, 100000), rng.randint(1, 65535 * 120)])
        D = 8 * rng.randint(1, 1024)
        E, sms = rng.randint(1, 256), rng.choice([1, 3, 8, 132, 148, 152, rng.randint(1, 2000)])
        assert rf.rf_selftest_moe_plan(T, D, E, sms) == 0, (T, D, E, sms)


def test_moe_plan_refused(rf):
    for args in [(0, 8, 64, 152), (1, 0, 64, 152), (1, 12, 64, 152), (1, 8, 0, 152),
                 (1, 8, 257, 152), (1, 8, 64, 0)]:
        assert rf.rf_selftest_moe_plan(*args) == -1, args
