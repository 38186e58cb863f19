"""skv_ideal_bits_noalloc: ideal bits without a caller workspace.

Some callers cannot allocate device memory at the point where they need the
ideal code length -- for instance a serving engine that reserved all free HBM
for its KV-cache pool at start-up, or a plugin running inside such an engine
without access to its allocator.  The no-allocation entry point keeps its
scratch in a fixed device array inside the library.  These tests check,
through the C ABI, that two calls in a row agree with skv_ideal_bits (the
workspace entry point) within the tolerance of the other GPU tests, with and
without the per-scalar output, and that an oversized shape is refused.
The file runs last so that it sees the library after every other test, and
it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import device_views, gpu_codec

pytestmark = pytest.mark.gpu

RTOL, ATOL = 1e-3, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("spec", [
    synth.WORKLOADS["tiny-bf16"],
    synth.WORKLOADS["qwen3-8b-e4m3"].scaled(name="noalloc-e4m3", L=2, H=2, T=300, D=64, Tb=128,
                                           G=4),
], ids=["bf16", "e4m3"])
def test_noalloc_matches_workspace_entry_point(spec):
    import lossless_kv_cache_fixed_gb300 as P
    w = synth.make(spec)
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    ref_tot, ref_ps = codec.ideal_bits(kv_d, mu_d, per_scalar=True)
    ref_ps = ref_ps.double().cpu().numpy()
    stream = P._stream_handle()
    for _ in range(2):
        ps = torch.full((codec.n,), float("nan"), dtype=torch.float32, device="cuda")
        rc, tot = P.skv_ideal_bits_noalloc(codec.params, codec.shape, kv_d.data_ptr(),
                                           mu_d.data_ptr(), ps.data_ptr(), stream)
        assert rc == P.SKV_OK, P.skv_strerror(rc)
        assert abs(tot - ref_tot) <= RTOL * abs(ref_tot)
        got = ps.double().cpu().numpy()
        assert np.all(np.abs(got - ref_ps) <= RTOL * np.abs(ref_ps) + ATOL)
        rc, tot2 = P.skv_ideal_bits_noalloc(codec.params, codec.shape, kv_d.data_ptr(),
                                            mu_d.data_ptr(), None, stream)
        assert rc == P.SKV_OK
        assert abs(tot2 - ref_tot) <= RTOL * abs(ref_tot)


def test_noalloc_rejects_oversized_shapes():
    import lossless_kv_cache_fixed_gb300 as P
    cap = P.skv_ideal_bits_noalloc_max_channels()
    assert cap >= 64 * 2 * 8 * 128          # every workload here fits
    heads = cap // (2 * 128) + 1             # one layer, head_dim 128: just over the limit
    params = P.SkvParams(P.SKV_E4M3, 256, 8, 0, 1 << 20, None, None)
    shape = P.SkvShape(1, 2, heads, 256, 128)
    rc, _ = P.skv_ideal_bits_noalloc(params, shape, 1 << 20, 1 << 20, None, None)
    assert rc == P.SKV_ERR_CAPACITY
