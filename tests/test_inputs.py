"""Synthetic-input generator: reproducible, slice-independent, shaped as stated."""
import numpy as np

import tq_inputs as ti


def test_streams_reproducible_and_distinct():
    a = ti.fp16_normal(ti.stream_seed(0, ti.K_ID, 0, 1), (64, 128))
    b = ti.fp16_normal(ti.stream_seed(0, ti.K_ID, 0, 1), (64, 128))
    c = ti.fp16_normal(ti.stream_seed(0, ti.K_ID, 0, 2), (64, 128))
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c)


def test_counter_form():
    full = ti.splitmix64(9, 100)
    np.testing.assert_array_equal(ti.splitmix64(9, 30, start=70), full[70:])


def test_outliers_and_lengths():
    w = ti.WORKLOADS["c3_turbo4v2_ragged"]
    L = w.lengths()
    assert L.shape == (8,) and L.min() >= 1024 and L.max() <= 8192
    o = w.outliers()
    assert len(o) == 4 and len(set(o.tolist())) == 4
    k = w.k_slice(0, 0, 4096).astype(np.float32)
    sd = k.std(0)
    assert np.all(sd[o] > 6) and np.median(np.delete(sd, o)) < 1.1
    assert ti.outlier_channels(96).size == 3


def test_kv_full_equals_slices():
    w = ti.Workload("t", 2, 4, 2, 64, 32, 4, 4, True)
    K = w.kv("k", threads=2)
    np.testing.assert_array_equal(K[1, 0], w.k_slice(1, 0))
    assert K.shape == (2, 2, 32, 64) and K.dtype == np.float16


def test_packed_bytes_of_long_context_workload():
    assert ti.WORKLOADS["c4_long_k8v3"].packed_kv_bytes() == 47_185_920
    assert ti.WORKLOADS["c2_llama3b"].packed_kv_bytes() == 4_325_376
    assert ti.WORKLOADS["c4_long_k8v3_d96"].packed_kv_bytes() == 35_651_584
