"""The input generator: reproducible, and its torch copy draws the same bytes."""
import numpy as np
import pytest

from quantized_moe_expert_sigmoid_gb300 import synth


def test_splitmix64_reference_values():
    # SplitMix64 with state 0 (Vigna's splitmix64.c: state += golden; mix):
    # first outputs 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4.
    out = synth.u64(np.uint64(0), 2, start=1)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4]


def test_streams_are_reproducible_and_distinct():
    a = synth.iq4nl_blocks(0, "up", 8, 256, 0, 1)
    b = synth.iq4nl_blocks(0, "up", 8, 256, 0, 1)
    c = synth.iq4nl_blocks(0, "up", 8, 256, 0, 2)
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_block_scale_range_and_nibbles_uniform():
    m = synth.iq4nl_blocks(1, "gate", 256, 1024)
    d = m[..., :2].copy().view(np.float16).astype(np.float64)
    assert d.min() >= 5e-4 * (1 - 2 ** -11) and d.max() <= 2e-3 * (1 + 2 ** -11)
    q = m[..., 2:]
    nib = np.concatenate([(q & 15).ravel(), (q >> 4).ravel()])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.95 * nib.size / 16 and counts.max() < 1.05 * nib.size / 16


def test_torch_copy_draws_identical_bytes():
    torch = pytest.importorskip("torch")
    for rows, cols, ids in ((4, 256, (0, 3)), (33, 96, (7,))):
        a = synth.iq4nl_blocks(5, "down", rows, cols, *ids)
        b = synth.iq4nl_blocks_torch(5, "down", rows, cols, *ids, device="cpu").numpy()
        assert np.array_equal(a, b)


def test_activation_rows_redraw_independently():
    att = np.zeros(4, np.int64)
    x0 = synth.activations(0, "x", 4, 64, att)
    att[2] = 1
    x1 = synth.activations(0, "x", 4, 64, att)
    assert np.array_equal(x0[[0, 1, 3]], x1[[0, 1, 3]]) and not np.array_equal(x0[2], x1[2])


def test_zipf_bias_prefers_low_ranks():
    b = synth.zipf_logit_bias(0, 512, 64)
    assert b.shape == (512, 64) and b.dtype == np.float32
    col = b.mean(axis=0)
    assert col.max() - col.min() > 1.0


def test_selection_bias_rows():
    b = synth.selection_bias(0, 64)
    m = synth.selection_bias(0, 64, 16)
    assert b.shape == (64,) and m.shape == (16, 64) and b.dtype == m.dtype == np.float32
    assert 0.05 < b.std() < 0.2 and not np.array_equal(m[0], b)
