"""The seeded input generators: SplitMix64 against its published output sequence."""
import numpy as np

from kv_cache_quantization_turbo_gb300 import workloads as W

GAMMA = 0x9E3779B97F4A7C15
# First outputs of SplitMix64 started from state 0 (Vigna's splitmix64.c):
# next() = mix(state += gamma), so the k-th output is mix((k+1) * gamma) = splitmix64(k * gamma).
PUBLISHED = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_published_sequence():
    counters = np.array([(k * GAMMA) % 2**64 for k in range(3)], dtype=np.uint64)
    assert [int(v) for v in W.splitmix64(counters)] == PUBLISHED


def test_signs_and_gaussians_shape_and_law():
    s = W.wht_signs(1, 128)
    assert s.dtype == np.int8 and set(np.unique(s)) <= {-1, 1}
    assert abs(int(s.sum())) < 40
    S = W.qjl_matrix(2, 128)
    assert S.dtype == np.float32 and S.shape == (128, 128)
    assert abs(float(S.mean())) < 0.03 and abs(float(S.std()) - 1.0) < 0.03
    # counter based: the d=64 table is not a prefix of the d=128 one, but the uniforms are
    np.testing.assert_array_equal(W.uniform53(2, 10), W.uniform53(2, 20)[:10])
    u = W.uniform53(3, 100000)
    assert u.min() > 0 and u.max() <= 1.0


def test_seq_lens_and_block_table():
    L = W.seq_lens_uniform(64, 1024, 16384, 0)
    assert L.min() >= 1024 and L.max() <= 16384
    bt, n = W.shuffled_block_table(L, 16, 0)
    used = bt[bt >= 0]
    assert len(np.unique(used)) == used.size == n
    assert all((bt[b] >= 0).sum() == (L[b] + 15) // 16 for b in range(64))


def test_decode_timing_cli_without_a_device():
    """The decode-timing module parses its recipes and refuses to run without CUDA (no CPU path)."""
    import pytest
    import torch
    from kv_cache_quantization_turbo_gb300 import decode_timing
    with pytest.raises(SystemExit):
        decode_timing.main(["--workload", "no-such-recipe"])
    if not torch.cuda.is_available():
        with pytest.raises(SystemExit, match="CUDA"):
            decode_timing.main(["--workload", "paged-batch64-turbo3", "--head-dim", "64"])
