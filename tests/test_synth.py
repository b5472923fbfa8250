"""The shared input generator: Philox4x32-10 against the published
known-answer vectors of its authors' reference implementation, and the
value mappings' basic statistics."""
import numpy as np

from synth import philox, workloads


def _one(ctr, key):
    out = philox.philox4x32_10(*[np.array([c], dtype=np.uint32) for c in ctr], *key)
    return [int(o[0]) for o in out]


def test_philox_known_answers():
    assert _one((0, 0, 0, 0), (0, 0)) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert _one((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2) == \
        [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert _one((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0)) == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_normal_mapping_statistics():
    x = philox.normal_f32(1, philox.STREAM_GRAD, 0, np.arange(400_000, dtype=np.uint64), 0.02)
    assert abs(float(x.mean())) < 2e-4 and abs(float(x.std()) / 0.02 - 1) < 0.01


def test_outliers_fraction():
    idx = np.arange(200_000, dtype=np.uint64)
    a = philox.grad_bf16(2, 0, idx, 1e-3)
    b = philox.grad_bf16(2, 0, idx, 1e-3, outlier_frac=0.01)
    frac = float(np.mean(a != b))
    assert 0.008 < frac < 0.012


def test_workload_sizes():
    assert workloads.tiny().psi == 37_248
    assert workloads.llama_layer().psi == 202_383_360
    assert workloads.llama3_layers().psi == 3_489_792_000
    assert workloads.llama3_8b().psi == 8_030_261_248
    ms = workloads.many_small()
    assert ms.n_params == 10_000 and sum(n < 100_000 for n in ms.numel) == 7500


def test_pool_offsets_disjoint_within_bucket():
    offs = workloads.pool_offsets([100, 1000, 37, 5000], 4, 30_000)
    lens = [128, 1024, 64, 5056]
    for row, L in zip(offs, lens):
        spans = sorted((o, o + L) for o in row)
        for (a, b), (c, d) in zip(spans, spans[1:]):
            assert b <= c
        assert all(o % 64 == 0 and o + L <= 30_000 for o in row)


def test_pool_offsets_exact_fit_without_wrap():
    offs = workloads.pool_offsets([40], 4, 256)
    assert offs == [[0, 64, 128, 192]]
