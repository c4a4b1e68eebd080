"""CPU check of the test helpers' bf16 decoding: widening bf16 to float64
through PyTorch gives the same value as the oracle's bit-pattern decoding
for every one of the 65536 bf16 bit patterns (NaN payloads aside)."""
import numpy as np
import torch

from oracle import moe_ref as ref
from _util import bf16_to_np64


def test_bf16_widening_equals_bit_decoding_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    got = bf16_to_np64(t)
    want = ref.bf16_to_f64(bits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
