"""GPU codec parity: the library's e4m3 encoder (the conversion the append
uses) against the oracle's on all 2^32 fp32 bit patterns, bit-exact.  This
also settles readings R1 (saturation) and R2 (signed zero) against the
hardware conversion."""
import numpy as np
import pytest
import torch

import oracle
from paged_fp8_kv_quantize_gb300 import abi

pytestmark = pytest.mark.gpu


def test_encode_all_fp32_bit_patterns():
    chunk = 1 << 28
    codes = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda").to(torch.int32)
        abi.e4m3_encode(bits.view(torch.float32), codes)
        got = codes.cpu().numpy()
        want = oracle.e4m3_encode_bits(np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32))
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (f"{bad.size} mismatches in chunk 0x{start:08x}; first bits 0x{start + int(bad[0]):08x}: "
                               f"gpu 0x{int(got[bad[0]]):02x} oracle 0x{int(want[bad[0]]):02x}")


def test_encode_ragged_length():
    x = torch.tensor([1.0, -2.0, 448.0, 1000.0, 0.0, -0.0, 2.0 ** -10], dtype=torch.float32, device="cuda")
    got = abi.e4m3_encode(x).cpu().numpy()
    assert list(got) == list(oracle.e4m3_encode(x.cpu().numpy()))
