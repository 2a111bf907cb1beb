"""Decode attention for callers that cannot allocate device memory.

Some callers of this library have no way to allocate GPU memory: a plugin whose
host framework owns every device buffer and grants it no workspace, a serving
loop whose memory budget is fixed at start-up, or a plain C caller without a
device allocator. For them, paged_decode_attention_bf16_noalloc keeps its
split-KV partials in a scratch array built into the library instead of a
caller-provided workspace. These checks call it through the C ABI and compare
it with the workspace entry point on the same inputs, over two calls in a row
(the scratch keeps the previous call's contents, which must not leak into the
next result).
"""
import numpy as np
import pytest

import synth
from gpu_util import bf16_close, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def a8w8():
    import w8a8_quantized_decode_gb300 as m
    m.build()
    return m


def _case(seed, B, Hq, Hkv, D, page, ctx):
    ctx = np.asarray(ctx, np.int32)
    bt, nblk = synth.paged_layout(seed, np.maximum(ctx, 1), page, spare_blocks=2)
    kc = synth.kv_cache(seed + 1, nblk, page, Hkv, D)
    vc = synth.kv_cache(seed + 2, nblk, page, Hkv, D)
    q = synth.bf16_normal(seed + 3, (B, Hq, D))
    return q, kc, vc, bt, ctx


def test_noalloc_matches_workspace_entry_on_two_calls(a8w8):
    import torch
    B, Hq, Hkv, D, page = 4, 40, 8, 128, 128
    # long contexts, so that the partials of several KV chunks live in the scratch
    for seed, ctx in ((11, [4096, 300, 1, 2049]), (12, [129, 3000, 64, 0])):
        q, kc, vc, bt, ctxa = _case(seed, B, Hq, Hkv, D, page, ctx)
        need = a8w8.attention_workspace_bytes(B, Hq, D, bt.shape[1] * page)
        assert 0 < need <= a8w8.NOALLOC_SCRATCH_BYTES
        args = [to_dev(q), to_dev(kc), to_dev(vc), to_dev(bt), to_dev(ctxa), page]
        ref = a8w8.paged_decode_attention_bf16(*args)
        got = a8w8.paged_decode_attention_bf16_noalloc(*args)
        torch.cuda.synchronize()
        g, r = to_host(got), to_host(ref)
        assert bf16_close(g, r, 2, 0.1).all()
        assert np.array_equal(g, r)        # same kernel and inputs: identical
        assert not g[np.asarray(ctxa) == 0].any()
    assert a8w8.read_device_errors() == 0


def test_noalloc_rejects_partials_larger_than_its_scratch(a8w8):
    # 64 requests x 64 heads x 128-token chunks of a 32768-token context need far
    # more than the built-in scratch: refused on the host, nothing launched
    fake = 0x10000
    st = a8w8.lib().paged_decode_attention_bf16_noalloc(
        fake, fake, fake, fake, fake, 64, 64, 8, 128, 128, 256, 300, 0.088, fake, None)
    assert st == a8w8.ERR_WORKSPACE
    assert b"scratch" in a8w8.lib().a8w8_last_error()
    assert a8w8.attention_workspace_bytes(64, 64, 128, 256 * 128) > a8w8.NOALLOC_SCRATCH_BYTES
