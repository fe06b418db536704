"""The seeded input generators: deterministic, with the stated shapes."""
import numpy as np

import oracle
import spmm_workloads as W


def test_generators_are_deterministic():
    a = W.bcsr_tiny()
    b = W.bcsr_tiny()
    assert np.array_equal(a.row_ptr, b.row_ptr) and np.array_equal(a.col_idx, b.col_idx)
    assert np.array_equal(a.vals, b.vals) and np.array_equal(a.B(), b.B())


def test_bcsr_tiny_shape():
    w = W.bcsr_tiny()
    assert (w.m, w.k, w.n, w.dtype, w.out_dtype) == (512, 512, 128, "f16", "f32")
    assert oracle.csr_check(w.m, w.k, w.row_ptr, w.col_idx) == 0
    # whole 64x64 blocks: every row holds a multiple of 64 entries
    assert np.all(np.diff(w.row_ptr) % 64 == 0)
    assert np.all((w.vals & 0x7FFF) != 0)


def test_bernoulli_density():
    rng = np.random.default_rng(1)
    rp, ci = W.bernoulli_pattern(rng, 2000, 3000, 0.01)
    assert oracle.csr_check(2000, 3000, rp, ci) == 0
    assert abs(len(ci) / 6e6 - 0.01) < 0.0005


def test_powerlaw_pattern_small():
    rng = np.random.default_rng(2)
    rp, ci = W.powerlaw_pattern(rng, 4096, 4096, 1.8, 1, 500, 64, 0.7)
    assert oracle.csr_check(4096, 4096, rp, ci) == 0
    L = np.diff(rp)
    assert L.min() >= 1 and L.max() <= 500


def test_block_pattern_exact_count():
    rng = np.random.default_rng(3)
    rp, ci = W.block_pattern(rng, 640, 320, 64, 64, keep_count=7)
    assert len(ci) == 7 * 64 * 64
    assert oracle.csr_check(640, 320, rp, ci) == 0


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], np.float32)
    b = W.f32_to_bf16_bits(x)
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020]
