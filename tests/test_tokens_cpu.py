"""int32 token files (gpt2_tokens_*): next-token batches checked element by
element against numpy slicing of the same file.  Host code only."""
import os

import numpy as np
import pytest

import transformer_lm_step_gpt_b300 as tl


def _write(path, arr):
    np.asarray(arr, dtype="<i4").tofile(path)


def test_batches_are_the_file_shifted_by_one(tmp_path):
    rng = np.random.default_rng(5)
    s = rng.integers(0, 50257, size=1000, dtype=np.int32)
    p = tmp_path / "toks.bin"
    _write(p, s)
    with tl.TokenFile(str(p)) as f:
        assert len(f) == 1000
        B, T = 3, 50
        pos = 0
        for _ in range(12):  # 12 * 150 > 1000: wraps around
            if pos + B * T + 1 > len(s):
                pos = 0
            x, y = f.next_batch(B, T)
            np.testing.assert_array_equal(x, s[pos:pos + B * T].reshape(B, T))
            np.testing.assert_array_equal(y, s[pos + 1:pos + B * T + 1].reshape(B, T))
            pos += B * T
        f.reset()
        x, y = f.next_batch(B, T)
        np.testing.assert_array_equal(x.ravel(), s[:B * T])


def test_exact_fit_and_errors(tmp_path):
    p = tmp_path / "small.bin"
    _write(p, np.arange(11))
    with tl.TokenFile(str(p)) as f:
        x, y = f.next_batch(2, 5)  # needs exactly 11 tokens
        np.testing.assert_array_equal(x.ravel(), np.arange(10))
        np.testing.assert_array_equal(y.ravel(), np.arange(1, 11))
        x, y = f.next_batch(2, 5)  # starts over
        np.testing.assert_array_equal(x.ravel(), np.arange(10))
        with pytest.raises(tl.GPT2Error) as e:
            f.next_batch(3, 4)  # 13 > 11 tokens
        assert e.value.code == -1
        with pytest.raises(tl.GPT2Error) as e:
            f.next_batch(0, 4)
        assert e.value.code == -1
    bad = tmp_path / "bad.bin"
    bad.write_bytes(b"\x01\x02\x03\x04\x05\x06")  # not a multiple of 4 bytes
    with pytest.raises(tl.GPT2Error) as e:
        tl.TokenFile(str(bad))
    assert e.value.code == -1
    with pytest.raises(tl.GPT2Error) as e:
        tl.TokenFile(str(tmp_path / "missing.bin"))
    assert e.value.code == -8  # GPT2_ERR_IO


def test_into_caller_buffers(tmp_path):
    s = np.arange(100, 200, dtype=np.int32)
    p = tmp_path / "t.bin"
    _write(p, s)
    x = np.zeros((2, 7), np.int32)
    y = np.zeros((2, 7), np.int32)
    with tl.TokenFile(str(p)) as f:
        f.next_batch(2, 7, x, y)
    np.testing.assert_array_equal(x.ravel(), s[:14])
    np.testing.assert_array_equal(y.ravel(), s[1:15])


def test_caller_buffers_are_checked_before_the_read(tmp_path):
    p = tmp_path / "toks.bin"
    _write(p, np.arange(200))
    with tl.TokenFile(str(p)) as f:
        x, y = np.empty((2, 8), np.int32), np.empty((2, 8), np.int32)
        f.next_batch(2, 8, x, y)                      # caller-owned buffers are filled in place
        np.testing.assert_array_equal(x.ravel(), np.arange(16))
        with pytest.raises(ValueError, match="15 elements, need 16"):
            f.next_batch(2, 8, np.empty(15, np.int32), y)
        with pytest.raises(TypeError, match="int64"):
            f.next_batch(2, 8, x, np.empty(16, np.int64))
        with pytest.raises(ValueError, match="contiguous"):
            f.next_batch(2, 8, np.empty((2, 16), np.int32)[:, ::2], y)
        x2, _ = f.next_batch(2, 8, x, y)              # the failed calls did not move the cursor
        np.testing.assert_array_equal(x2.ravel(), np.arange(16, 32))
