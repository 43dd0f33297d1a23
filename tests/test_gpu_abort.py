"""The decode kernels' abort path, exercised without any fault: the
PFKV_FLAG_TEST_WITHHOLD hook makes the first CTA's page loader withhold its
first work item, so the other warps' bounded waits run out (about 2 s).
Every request must report TIMEOUT, the call must return, and the next call
on the same context must match the oracle."""
import numpy as np
import pytest

from gpu_helpers import DeviceCase, assert_close
from oracle_helpers import oracle_cache
from paged_fp8_kv_quantize_gb300 import abi, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [abi.DTYPE_FP8_E4M3, abi.DTYPE_BF16])
def test_withheld_item_times_out_and_context_stays_usable(dtype):
    lens = [300, 2000, 17, 4097, 1, 700]
    w = synth.make("abort", 950, batch=len(lens), q_heads=32, kv_heads=8, head_dim=128, page_size=16,
                   seq_lens=lens, outlier_p=0.01)
    run = DeviceCase(w, dtype)
    _, st = run.decode(flags=abi.FLAG_TAG_CHECK | abi.FLAG_TEST_WITHHOLD)
    assert np.all(st & abi.ST_TIMEOUT), st
    out, st2 = run.decode(flags=abi.FLAG_TAG_CHECK)
    ref, _ = oracle_cache(w, dtype)
    o_ref, st_ref = ref.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale,
                               flags=abi.FLAG_TAG_CHECK, threads=8)
    assert np.array_equal(st2, st_ref)
    assert_close(out, o_ref, "decode after an aborted call")


def test_latent_withheld_item_times_out_and_context_stays_usable():
    lens = [4096, 4096, 3000, 5000]  # enough pages for one balanced range per CTA
    w = synth.make("abort_lat", 951, batch=len(lens), q_heads=64, kv_heads=1, head_dim=576, v_head_dim=512,
                   kv_shared=True, page_size=64, seq_lens=lens, scale_mode=synth.PER_TOKEN,
                   softmax_scale=1.0 / 24.0)
    run = DeviceCase(w)
    _, st = run.decode(flags=abi.FLAG_TAG_CHECK | abi.FLAG_TEST_WITHHOLD)
    assert np.all(st & abi.ST_TIMEOUT), st
    out, st2 = run.decode(flags=abi.FLAG_TAG_CHECK)
    ref, _ = oracle_cache(w)
    o_ref, st_ref = ref.decode(w.q, w.seq_lens, w.block_table, w.block_tags, w.softmax_scale,
                               flags=abi.FLAG_TAG_CHECK, threads=8)
    assert np.array_equal(st2, st_ref)
    assert_close(out, o_ref, "latent decode after an aborted call")
