"""skv_ideal_bits_noalloc: ideal bits without a caller workspace.

Some callers cannot allocate device memory at the point where they need the
ideal code length -- for instance a serving engine that reserved all free HBM
for its KV-cache pool at start-up, or a plugin running inside such an engine
without access to its allocator.  The no-allocation entry point keeps its
scratch in a fixed device array inside the library.  These tests check,
through the C ABI, that two calls in a row agree with the oracle and with
skv_ideal_bits (the workspace entry point) within the tolerance of the other
GPU tests, with and without the per-scalar output; that a shape at exactly the
advertised sigma limit is accepted and correct; and that one entry over it is
refused.  Every call gets real device buffers of the right size, so no
ordering of the library's checks can launch a kernel on a bad pointer.
The file runs last so that it sees the library after every other test, and
it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import device_views, gpu_codec, host_views, oracle_model

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
def test_noalloc_matches_oracle_and_workspace_entry_point(spec, oracle_mod):
    import lossless_kv_cache_fixed_gb300 as P
    w = synth.make(spec)
    codec = gpu_codec(w)
    kv_d, mu_d = device_views(w)
    kv_h, mu_h = host_views(w)
    ora_tot, ora_ps = oracle_mod.ideal_bits(oracle_model(oracle_mod, w), kv_h, mu_h,
                                            per_scalar=True)
    ref_tot, ref_ps = codec.ideal_bits(kv_d, mu_d, per_scalar=True)
    ref_ps = ref_ps.double().cpu().numpy()
    stream = P._stream_handle()
    for _ in range(2):
        ps = torch.full((codec.n,), float("nan"), dtype=torch.float32, device="cuda")
        rc, tot = P.skv_ideal_bits_noalloc(codec.params, codec.shape, kv_d.data_ptr(),
                                           mu_d.data_ptr(), ps.data_ptr(), stream)
        assert rc == P.SKV_OK, P.skv_strerror(rc)
        got = ps.double().cpu().numpy()
        # against the oracle directly, and against the workspace entry point
        assert np.all(np.abs(got - ora_ps) <= RTOL * np.abs(ora_ps) + ATOL)
        assert abs(tot - ora_tot) <= RTOL * abs(ora_tot)
        assert np.all(np.abs(got - ref_ps) <= RTOL * np.abs(ref_ps) + ATOL)
        assert abs(tot - ref_tot) <= RTOL * abs(ref_tot)
        rc, tot2 = P.skv_ideal_bits_noalloc(codec.params, codec.shape, kv_d.data_ptr(),
                                            mu_d.data_ptr(), None, stream)
        assert rc == P.SKV_OK
        assert abs(tot2 - ora_tot) <= RTOL * abs(ora_tot)


def _e4m3_buffers(heads, head_dim, tokens):
    """Real device buffers of an e4m3 cache with one layer: KV codes, mu and sigma."""
    n = 2 * heads * tokens * head_dim
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    codes = torch.randint(0, 0x7F, (n,), generator=g, device="cuda", dtype=torch.uint8)
    kv = codes | (torch.randint(0, 2, (n,), generator=g, device="cuda", dtype=torch.uint8) << 7)
    mu = (torch.randn(n, generator=g, device="cuda") * 40.0).to(torch.bfloat16).view(torch.int16)
    sigma = torch.full((2 * heads * head_dim,), 3.0, dtype=torch.float32, device="cuda")
    return kv, mu, sigma


def test_noalloc_sigma_limit_boundary():
    import lossless_kv_cache_fixed_gb300 as P
    cap = P.skv_ideal_bits_noalloc_max_channels()
    assert cap >= 64 * 2 * 8 * 128          # every workload here fits
    stream = P._stream_handle()
    # exactly at the limit, with enough tokens that the kernel runs its largest
    # grid (the partial-sum array at its maximum size)
    D = 32
    assert cap % (2 * D) == 0
    H = cap // (2 * D)
    T = 40
    kv, mu, sigma = _e4m3_buffers(H, D, T)
    params = P.SkvParams(P.SKV_E4M3, 16, 4, 0, sigma.data_ptr(), None, None)
    shape = P.SkvShape(1, 2, H, T, D)
    assert 2 * H * T * D // 8 // 256 >= 4096
    rc, tot = P.skv_ideal_bits_noalloc(params, shape, kv.data_ptr(), mu.data_ptr(), None, stream)
    assert rc == P.SKV_OK, P.skv_strerror(rc)
    ws = torch.empty(P.skv_workspace_bytes(params, shape, P.SKV_OP_IDEAL_BITS), dtype=torch.uint8,
                     device="cuda")
    rc, ref = P.skv_ideal_bits(params, shape, kv.data_ptr(), mu.data_ptr(), None,
                               ws.data_ptr(), ws.numel(), stream)
    assert rc == P.SKV_OK
    assert abs(tot - ref) <= RTOL * abs(ref)
    # one (layer, kv, head) row of channels over the limit: refused before any launch
    kv2, mu2, sigma2 = _e4m3_buffers(H + 1, D, 1)
    params2 = P.SkvParams(P.SKV_E4M3, 16, 4, 0, sigma2.data_ptr(), None, None)
    shape2 = P.SkvShape(1, 2, H + 1, 1, D)
    rc, _ = P.skv_ideal_bits_noalloc(params2, shape2, kv2.data_ptr(), mu2.data_ptr(), None, stream)
    assert rc == P.SKV_ERR_CAPACITY
