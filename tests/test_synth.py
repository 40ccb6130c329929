"""The shared input generators: value distributions and the sentinel fill."""
import numpy as np
import pytest

import synth


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100_000, dtype=np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8]  # ties to even, both directions
    ours = synth.bf16_bits_from_f32(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_fp8_codes_exclude_nan():
    rng = np.random.default_rng(1)
    b = synth.fp8_e4m3_bytes(rng, 500_000)
    counts = np.bincount(b, minlength=256)
    assert counts[0x7F] == 0 and counts[0xFF] == 0
    assert np.count_nonzero(counts) == 254


def test_splitmix64_published_values():
    # Vigna's splitmix64 with state 0: the first outputs of the generator are
    # splitmix64(0), splitmix64(0x9E3779B97F4A7C15), ... (its published test
    # sequence starts 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4).
    out = synth.splitmix64_np(np.array([0, 0x9E3779B97F4A7C15], dtype=np.uint64))
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_sentinel_torch_matches_numpy():
    torch = pytest.importorskip("torch")
    n = 8 * 5000 + 16
    buf = torch.empty(n, dtype=torch.uint8)
    synth.fill_sentinel_torch(buf, 1234, chunk_words=777)
    ref = synth.sentinel_bytes(1234, 0, n)
    assert np.array_equal(buf.numpy(), ref)
    # any sub-range and any row set agree with the whole
    assert np.array_equal(synth.sentinel_bytes(1234, 13, 101), ref[13:114])
    rows = synth.sentinel_rows(1234, np.array([0, 64, 4096]), 64)
    assert np.array_equal(rows[2], ref[4096:4160])


def test_workload_shapes():
    s3 = synth.SHAPES[3]
    slots, pages = synth.prefill_slots(s3)
    assert slots.size == 32768 and pages.shape == (16, 32)
    assert np.count_nonzero(slots < 0) == round(0.02 * 32768)
    assert len(set(pages.reshape(-1).tolist())) == 512 and pages.min() >= 1
    s4 = synth.SHAPES[4]
    st, g = synth.swa_batch(s4)
    assert st.size == 512 and g.total == 512 * 128
    assert len(set(g.block_table.reshape(-1).tolist())) == 2560
    s1 = synth.SHAPES[1]
    sl = synth.store_slots(s1, 0)
    assert sl.size == 100 and np.count_nonzero(sl < 0) == 5
    valid = sl[sl >= 0]
    assert valid.min() >= 4 and valid.max() < 256 and len(set(valid.tolist())) == 95
    g1 = synth.gather_batch(s1)
    assert g1.block_table.shape == (1, 8) and g1.total == 32
